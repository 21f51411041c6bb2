// Non-causal multi-head softmax attention, O = softmax(Q K^T / sqrt(hd)) V,
// flash-style: one CTA per (64 query rows, head, batch), 4 warps of 16 rows,
// K/V tiles of 64 keys double-buffered in shared memory with cp.async,
// online softmax in fp32 with quad-shuffle row max / row sum, exp2 with the
// scale folded into log2(e) / sqrt(hd).  Head dims that are not a multiple
// of 16 (72) are zero-padded to the next multiple of 16 in shared memory, so
// the padded columns add nothing to Q K^T and are dropped from O.  Keys past
// nk are masked to -inf; query rows past nq are not stored.
//
// This kernel issues mma.sync m16n8k16 (bf16 in, fp32 accumulate); it serves
// the head dims the tcgen05 kernel in attention_tc.cu does not (it takes 64,
// 72, 80 and 128).
#include <cuda_bf16.h>

#include <cstdlib>
#include <string>

#include "internal.h"
#include "ptx.cuh"

namespace dlo {

namespace {

constexpr int BQ = 64;
constexpr int BKV = 64;
constexpr int kWarps = 4;

template <int HDP>
struct AttnSmem {
    static constexpr int PITCH = HDP + 8;                 // elements; +16 B breaks bank conflicts
    static constexpr int TILE = BQ * PITCH;               // elements per 64-row tile
    static constexpr int BYTES = (TILE + 4 * TILE) * 2;   // Q, K[2], V[2]
};

// Copy rows r0 .. r0+63 of one head (hd columns) into a padded smem tile;
// missing rows and the padding columns are zero.
template <int HDP>
__device__ __forceinline__ void load_tile(__nv_bfloat16* tile, const __nv_bfloat16* base, int r0,
                                          int nrows, int ld, int hd) {
    constexpr int CH = HDP / 8;   // 16-byte chunks per padded row
    const int hd8 = hd / 8;
    for (int i = threadIdx.x; i < BQ * CH; i += kWarps * 32) {
        const int r = i / CH, c = i % CH;
        const int gr = r0 + r;
        const bool valid = gr < nrows && c < hd8;
        const __nv_bfloat16* src = valid ? base + static_cast<size_t>(gr) * ld + c * 8 : base;
        cp_async16(smem_u32(tile + r * AttnSmem<HDP>::PITCH + c * 8), src, valid ? 16u : 0u);
    }
}

template <int HDP>
__global__ void __launch_bounds__(kWarps * 32)
    attn_fwd_kernel(const __nv_bfloat16* __restrict__ Q, const __nv_bfloat16* __restrict__ K,
                    const __nv_bfloat16* __restrict__ V, __nv_bfloat16* __restrict__ O, int hd,
                    int nq, int nk, int ldq, int ldk, int ldv, int ldo, float scale_log2) {
    pdl_wait();
    pdl_launch_dependents();
    using S = AttnSmem<HDP>;
    constexpr int PITCH = S::PITCH;
    constexpr int KSTEPS = HDP / 16;     // k-steps of Q K^T
    constexpr int NT_O = HDP / 8;        // n-tiles of O
    extern __shared__ __align__(16) __nv_bfloat16 sm[];
    __nv_bfloat16* sQ = sm;
    __nv_bfloat16* sK = sm + S::TILE;            // 2 buffers
    __nv_bfloat16* sV = sm + 3 * S::TILE;        // 2 buffers

    const int b = blockIdx.z, h = blockIdx.y, q0 = blockIdx.x * BQ;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const __nv_bfloat16* Qb = Q + static_cast<size_t>(b) * nq * ldq + h * hd;
    const __nv_bfloat16* Kb = K + static_cast<size_t>(b) * nk * ldk + h * hd;
    const __nv_bfloat16* Vb = V + static_cast<size_t>(b) * nk * ldv + h * hd;

    load_tile<HDP>(sQ, Qb, q0, nq, ldq, hd);
    cp_async_commit();
    load_tile<HDP>(sK, Kb, 0, nk, ldk, hd);
    load_tile<HDP>(sV, Vb, 0, nk, ldv, hd);
    cp_async_commit();

    // Q fragments of this warp's 16 rows, kept in registers
    cp_async_wait<1>();
    __syncthreads();
    uint32_t qf[KSTEPS][4];
    {
        const int r = warp * 16 + (lane & 15);
        const int c = (lane >> 4) * 8;
#pragma unroll
        for (int ks = 0; ks < KSTEPS; ++ks)
            ldsm_x4(smem_u32(sQ + r * PITCH + ks * 16 + c), qf[ks][0], qf[ks][1], qf[ks][2],
                    qf[ks][3]);
    }

    float o[NT_O][4];
#pragma unroll
    for (int j = 0; j < NT_O; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;   // rows g and g+8

    const int ntiles = (nk + BKV - 1) / BKV;
    for (int t = 0; t < ntiles; ++t) {
        const int buf = t & 1;
        cp_async_wait<0>();
        __syncthreads();
        if (t + 1 < ntiles) {
            load_tile<HDP>(sK + (buf ^ 1) * S::TILE, Kb, (t + 1) * BKV, nk, ldk, hd);
            load_tile<HDP>(sV + (buf ^ 1) * S::TILE, Vb, (t + 1) * BKV, nk, ldv, hd);
        }
        cp_async_commit();
        const __nv_bfloat16* tK = sK + buf * S::TILE;
        const __nv_bfloat16* tV = sV + buf * S::TILE;

        // S = Q K^T : 16 rows x 64 keys per warp, 8 n-tiles of 8 keys
        float s[8][4];
#pragma unroll
        for (int j = 0; j < 8; ++j) s[j][0] = s[j][1] = s[j][2] = s[j][3] = 0.f;
#pragma unroll
        for (int ks = 0; ks < KSTEPS; ++ks) {
#pragma unroll
            for (int jp = 0; jp < 4; ++jp) {     // pairs of key n-tiles
                const int mi = lane >> 3;
                const int key = jp * 16 + (mi >> 1) * 8 + (lane & 7);
                const int dim = ks * 16 + (mi & 1) * 8;
                uint32_t b0, b1, b2, b3;
                ldsm_x4(smem_u32(tK + key * PITCH + dim), b0, b1, b2, b3);
                mma_bf16_16816(s[2 * jp], qf[ks], b0, b1);
                mma_bf16_16816(s[2 * jp + 1], qf[ks], b2, b3);
            }
        }
        // mask keys past nk (only the last tile can have them)
        const int kbase = t * BKV;
        if (kbase + BKV > nk) {
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int c = kbase + j * 8 + (lane & 3) * 2;
                if (c >= nk) s[j][0] = s[j][2] = -INFINITY;
                if (c + 1 >= nk) s[j][1] = s[j][3] = -INFINITY;
            }
        }
        // online softmax (log2 domain)
        float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            mx0 = fmaxf(mx0, fmaxf(s[j][0], s[j][1]));
            mx1 = fmaxf(mx1, fmaxf(s[j][2], s[j][3]));
        }
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xFFFFFFFFu, mx0, 1));
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xFFFFFFFFu, mx0, 2));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xFFFFFFFFu, mx1, 1));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xFFFFFFFFu, mx1, 2));
        const float mn0 = fmaxf(m0, mx0 * scale_log2);
        const float mn1 = fmaxf(m1, mx1 * scale_log2);
        const float c0 = exp2f(m0 - mn0), c1 = exp2f(m1 - mn1);
        m0 = mn0;
        m1 = mn1;
        float rs0 = 0.f, rs1 = 0.f;
        uint32_t pf[4][4];   // P as A fragments, one per 16-key k-step
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const float p0 = exp2f(s[j][0] * scale_log2 - mn0);
            const float p1 = exp2f(s[j][1] * scale_log2 - mn0);
            const float p2 = exp2f(s[j][2] * scale_log2 - mn1);
            const float p3 = exp2f(s[j][3] * scale_log2 - mn1);
            rs0 += p0 + p1;
            rs1 += p2 + p3;
            pf[j >> 1][(j & 1) * 2 + 0] = pack_bf16x2(p0, p1);
            pf[j >> 1][(j & 1) * 2 + 1] = pack_bf16x2(p2, p3);
        }
        rs0 += __shfl_xor_sync(0xFFFFFFFFu, rs0, 1);
        rs0 += __shfl_xor_sync(0xFFFFFFFFu, rs0, 2);
        rs1 += __shfl_xor_sync(0xFFFFFFFFu, rs1, 1);
        rs1 += __shfl_xor_sync(0xFFFFFFFFu, rs1, 2);
        l0 = l0 * c0 + rs0;
        l1 = l1 * c1 + rs1;
#pragma unroll
        for (int j = 0; j < NT_O; ++j) {
            o[j][0] *= c0;
            o[j][1] *= c0;
            o[j][2] *= c1;
            o[j][3] *= c1;
        }
        // O += P V : k-steps of 16 keys, n-tiles of 8 dims (pairs per ldmatrix)
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) {
#pragma unroll
            for (int jp = 0; jp < NT_O / 2; ++jp) {
                const int mi = lane >> 3;
                const int key = ks * 16 + (mi & 1) * 8 + (lane & 7);
                const int dim = jp * 16 + (mi >> 1) * 8;
                uint32_t b0, b1, b2, b3;
                ldsm_x4_trans(smem_u32(tV + key * PITCH + dim), b0, b1, b2, b3);
                // reorder A fragment: pf[ks] holds {tile 2ks (c0c1), tile 2ks (c2c3),
                // tile 2ks+1 (c0c1), tile 2ks+1 (c2c3)}
                const uint32_t a[4] = {pf[ks][0], pf[ks][1], pf[ks][2], pf[ks][3]};
                mma_bf16_16816(o[2 * jp], a, b0, b1);
                mma_bf16_16816(o[2 * jp + 1], a, b2, b3);
            }
        }
    }
    cp_async_wait<0>();

    // normalise and store rows g, g+8 of this warp
    const float inv0 = 1.f / l0, inv1 = 1.f / l1;
    const int g = lane >> 2, tq = lane & 3;
    const int r0 = q0 + warp * 16 + g, r1 = r0 + 8;
    __nv_bfloat16* Ob = O + static_cast<size_t>(b) * nq * ldo + h * hd;
#pragma unroll
    for (int j = 0; j < NT_O; ++j) {
        const int d = j * 8 + tq * 2;
        if (d < hd) {
            if (r0 < nq)
                *reinterpret_cast<uint32_t*>(Ob + static_cast<size_t>(r0) * ldo + d) =
                    pack_bf16x2(o[j][0] * inv0, o[j][1] * inv0);
            if (r1 < nq)
                *reinterpret_cast<uint32_t*>(Ob + static_cast<size_t>(r1) * ldo + d) =
                    pack_bf16x2(o[j][2] * inv1, o[j][3] * inv1);
        }
    }
}

template <int HDP>
cudaError_t run(const void* Q, const void* K, const void* V, void* O, int batch, int heads, int hd,
                int nq, int nk, int ldq, int ldk, int ldv, int ldo, cudaStream_t s,
                unsigned long long* launches) {
    constexpr int bytes = AttnSmem<HDP>::BYTES;
    static bool attr = false;
    if (!attr) {
        cudaError_t e = cudaFuncSetAttribute(attn_fwd_kernel<HDP>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
        if (e != cudaSuccess) return e;
        attr = true;
    }
    const float scale_log2 = 1.4426950408889634f / sqrtf(static_cast<float>(hd));
    dim3 grid((nq + BQ - 1) / BQ, heads, batch);
    cudaError_t le_ = launch_k(attn_fwd_kernel<HDP>, grid, kWarps * 32, bytes, s, static_cast<const __nv_bfloat16*>(Q), static_cast<const __nv_bfloat16*>(K),
        static_cast<const __nv_bfloat16*>(V), static_cast<__nv_bfloat16*>(O), hd, nq, nk, ldq, ldk,
        ldv, ldo, scale_log2);
    ++*launches;
    return le_ != cudaSuccess ? le_ : cudaGetLastError();
}

}  // namespace

cudaError_t launch_attention(const void* Q, const void* K, const void* V, void* O, int batch,
                             int heads, int hd, int nq, int nk, int ldq, int ldk, int ldv, int ldo,
                             int* err, cudaStream_t s, unsigned long long* launches) {
    if (nq <= 0 || batch <= 0 || heads <= 0) return cudaSuccess;
    if (nk <= 0) return cudaErrorInvalidValue;
    static int force_sync = -1;
    if (force_sync < 0) {
        const char* e = std::getenv("DLO_ATTN");
        force_sync = (e && std::string(e) == "sync") ? 1 : 0;
    }
    if (!force_sync && attention_tc_supported(hd))
        return launch_attention_tc(Q, K, V, O, batch, heads, hd, nq, nk, ldq, ldk, ldv, ldo, err, s,
                                   launches);
    const int hdp = (hd + 15) / 16 * 16;
    switch (hdp) {
        case 16: return run<16>(Q, K, V, O, batch, heads, hd, nq, nk, ldq, ldk, ldv, ldo, s, launches);
        case 32: return run<32>(Q, K, V, O, batch, heads, hd, nq, nk, ldq, ldk, ldv, ldo, s, launches);
        case 48: return run<48>(Q, K, V, O, batch, heads, hd, nq, nk, ldq, ldk, ldv, ldo, s, launches);
        case 64: return run<64>(Q, K, V, O, batch, heads, hd, nq, nk, ldq, ldk, ldv, ldo, s, launches);
        case 80: return run<80>(Q, K, V, O, batch, heads, hd, nq, nk, ldq, ldk, ldv, ldo, s, launches);
        case 96: return run<96>(Q, K, V, O, batch, heads, hd, nq, nk, ldq, ldk, ldv, ldo, s, launches);
        case 112: return run<112>(Q, K, V, O, batch, heads, hd, nq, nk, ldq, ldk, ldv, ldo, s, launches);
        case 128: return run<128>(Q, K, V, O, batch, heads, hd, nq, nk, ldq, ldk, ldv, ldo, s, launches);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace dlo
