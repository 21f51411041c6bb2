// Non-causal multi-head attention on the 5th-generation tensor cores.
// O = softmax(Q K^T / sqrt(hd)) V for every head dim that is a multiple of 8
// up to 128.  Q, K and V tiles are whole 64-column blocks (one for hd <= 64,
// two for hd > 80); a head dim of 64 + t (t <= 16, e.g. 72) instead adds a
// 16-column tail block loaded with the 32-byte swizzle.  TMA fills the box
// columns past hd with zeros (a 4-D tensor map [batch, rows, heads, hd] ends
// each head at hd), so the padded columns add nothing to Q K^T and are
// dropped from O.
//
// One CTA per (128 query rows, head, batch); 6 warps:
//   warp 0      TMA: the Q tile once, then K_j and V_j tiles of 128 keys into
//               one ring stage, both completing one barrier (the MMA issuer
//               waits once per tile); rows past a batch's end are zero-filled
//   warp 1      MMA issuer (one thread): S_j = Q K_j^T into one of two TMEM S
//               buffers (128 fp32 columns each), and O += P_j V_j into the TMEM
//               O accumulator; issue order S_0, S_1, PV_0, S_2, PV_1, ... so the
//               tensor core computes S_{j+1} while the softmax warps work on S_j
//   warps 2..5  softmax, one thread per query row (its TMEM lane): load S_j,
//               mask keys past nk, running max in the log2 domain, p = 2^(s -
//               m), row sum, P_j as bf16 pairs over the first 64 columns of
//               its own S buffer in TMEM (P V reads A from tensor memory).
//               The reference max only moves
//               when a row's max grows by more than 8 (a factor 256), and only
//               then is that row's O rescaled in TMEM (ld, scale, st) -- the
//               p values stay below 2^8, which bf16 and fp32 hold exactly in
//               range.  At the end O / l is written as bf16.
// V is the B operand of P V in its natural [key][dim] layout, i.e. MN-major
// (dims contiguous): 64-dim blocks of 128-byte rows, one row per key.
//
// DUO (head dims up to 80): two CTAs share an SM.  Each holds one S buffer
// and O in 256 TMEM columns and two K/V stages in ~100 KB of shared memory;
// its MMAs run S_j, PV_j, S_{j+1}, ... and the other CTA's softmax fills the
// tensor core while this one's runs.  A grid of 1.7 waves of single CTAs then
// fits in one wave.
//
// Every mbarrier wait is bounded; a wait that runs out sets the error word
// and the abort flag, every role leaves its loop, in-flight TMA loads and
// MMAs are drained (bounded) and TMEM is freed.
#include <cuda.h>
#include <cuda_bf16.h>

#include <cstdlib>

#include "internal.h"
#include "ptx.cuh"

namespace dlo {

namespace {

constexpr int TQ = 128;          // query rows per CTA (MMA M, TMEM lanes)
constexpr int TK = 128;          // keys per tile
constexpr int kThreadsA = 192;

template <int NB, bool TAIL, bool DUO = false>
struct AttnPlan {
    static constexpr int HDP = NB * 64 + (TAIL ? 16 : 0);   // padded head dim
    static constexpr int BLK = 128 * 128;                   // 128 rows x 128 B (64 cols)
    static constexpr int TBLK = TAIL ? 128 * 32 : 0;        // 128 rows x 32 B (16 cols)
    static constexpr int TILE = NB * BLK + TBLK;            // one Q, K or V tile
    // K/V ring depth: three stages when they fit next to Q in shared memory
    // (DUO: two, so two CTAs fit on one SM)
    static constexpr int STAGES = DUO ? 2 : (TILE * 7 + 2048 <= 227 * 1024) ? 3 : 2;
    static constexpr int Q_OFF = 0;
    static constexpr int K_OFF = Q_OFF + TILE;              // STAGES stages
    static constexpr int V_OFF = K_OFF + STAGES * TILE;     // STAGES stages
    static constexpr int BAR_OFF = V_OFF + STAGES * TILE;
    // q_full, kv_full[3], k_empty[3], 3 spare, v_empty[3], s_full[2], p_full,
    // pv_done, drain
    static constexpr int NBARS = 1 + 12 + 2 + 3;
    static constexpr int TMEM_SLOT_OFF = BAR_OFF + NBARS * 8;
    static constexpr int ABORT_OFF = TMEM_SLOT_OFF + 4;
    static constexpr int USED = ABORT_OFF + 4 + 1024;
    // single CTAs: at least 116 KB, so one CTA per SM owns all 512 TMEM
    // columns; DUO: two CTAs of 256 columns each
    static constexpr int BYTES = DUO ? USED : (USED > 118784 ? USED : 118784);
    static constexpr uint32_t TMEM_COLS = DUO ? 256 : 512;
    static constexpr int SBUF = DUO ? 1 : 2;           // S buffers (128 columns each, from 0)
    static constexpr uint32_t O_COL = SBUF * 128;
    static_assert(!DUO || (NB == 1 && 2 * (USED + 1024) <= 228 * 1024), "DUO: two CTAs per SM");
};

struct AttnMaps {
    CUtensorMap q, k, v;        // 64-column boxes, 128-byte swizzle
    CUtensorMap qt, kt, vt;     // 16-column tail boxes, 32-byte swizzle
};

template <int NB, bool TAIL>
__device__ __forceinline__ void load_tile(uint32_t dst, const CUtensorMap* main,
                                          const CUtensorMap* tail, int h, int row0, int b,
                                          uint32_t bar) {
    using P = AttnPlan<NB, TAIL>;   // BLK and TBLK do not depend on DUO
#pragma unroll
    for (int blk = 0; blk < NB; ++blk) tma_load_4d(dst + blk * P::BLK, main, blk * 64, h, row0, b, bar);
    if constexpr (TAIL) tma_load_4d(dst + NB * P::BLK, tail, NB * 64, h, row0, b, bar);
}

template <int NB, bool TAIL, bool DUO>
__global__ void __launch_bounds__(kThreadsA, DUO ? 2 : 1)
    attn_tc_kernel(const __grid_constant__ AttnMaps maps, __nv_bfloat16* __restrict__ O, int hd,
                   int nq, int nk, int ldo, float scale_log2, int* err) {
    using P = AttnPlan<NB, TAIL, DUO>;
    constexpr int HDP = P::HDP;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const uint32_t sb = smem_u32(smem);
    const uint32_t bar = sb + P::BAR_OFF;
    const uint32_t q_full = bar;
    const uint32_t kv_full = bar + 8, k_empty = bar + 32;
    const uint32_t v_empty = bar + 80;
    const uint32_t s_full = bar + 104;
    const uint32_t p_full = bar + 120, pv_done = bar + 128, drain = bar + 136;
    constexpr int NS = P::STAGES;
    volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(smem + P::TMEM_SLOT_OFF);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + P::ABORT_OFF);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int qt = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int ntiles = (nk + TK - 1) / TK;

    if (threadIdx.x == 0) {
        mbar_init(q_full, 1);
        for (int i = 0; i < NS; ++i) {
            mbar_init(kv_full + 8 * i, 1);
            mbar_init(k_empty + 8 * i, 1);
            mbar_init(v_empty + 8 * i, 1);
        }
        for (int i = 0; i < 2; ++i) mbar_init(s_full + 8 * i, 1);
        mbar_init(p_full, 4);
        mbar_init(pv_done, 1);
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_mbar_init();
        tma_prefetch_desc(&maps.q);
        tma_prefetch_desc(&maps.k);
        tma_prefetch_desc(&maps.v);
    }
    if (warp == 1) {
        tmem_alloc(sb + P::TMEM_SLOT_OFF, P::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    pdl_wait();                 // predecessor's outputs complete and visible
    pdl_launch_dependents();

    auto fail = [&]() {
        *abort_flag = 1;
        if (err) atomicExch(err, 1);
    };

    if (warp == 0 && lane == 0) {
        // ---------------- TMA producer
        bool ok = true;
        uint32_t issued = 0;      // stages with a load in flight
        uint32_t par = 0;         // parity of that load's phase
        mbar_arrive_expect_tx(q_full, P::TILE);
        load_tile<NB, TAIL>(sb + P::Q_OFF, &maps.q, &maps.qt, h, qt * TQ, b, q_full);
        for (int j = 0; ok && j < ntiles; ++j) {
            const int st = j % NS;
            const uint32_t ph = (j / NS) & 1;
            // the stage's K is free after S_{j-NS}, its V after PV_{j-NS}
            if (!mbar_wait(k_empty + 8 * st, ph ^ 1, abort_flag) ||
                !mbar_wait(v_empty + 8 * st, ph ^ 1, abort_flag)) {
                fail();
                ok = false;
                break;
            }
            mbar_arrive_expect_tx(kv_full + 8 * st, 2 * P::TILE);
            load_tile<NB, TAIL>(sb + P::K_OFF + st * P::TILE, &maps.k, &maps.kt, h, j * TK, b, kv_full + 8 * st);
            load_tile<NB, TAIL>(sb + P::V_OFF + st * P::TILE, &maps.v, &maps.vt, h, j * TK, b, kv_full + 8 * st);
            issued |= 1u << st;
            par = (par & ~(1u << st)) | (ph << st);
        }
        if (!ok || *abort_flag) {
            mbar_wait(q_full, 0, nullptr);
            for (int i = 0; i < NS; ++i)
                if (issued & (1u << i)) mbar_wait(kv_full + 8 * i, (par >> i) & 1u, nullptr);
        }
    } else if (warp == 1 && lane == 0) {
        // ---------------- MMA issuer
        constexpr uint32_t idesc_s = idesc_bf16_f32(TQ, TK);
        constexpr uint32_t idesc_o = idesc_bf16_f32(TQ, NB * 64, true);
        constexpr uint32_t idesc_ot = idesc_bf16_f32(TQ, 16, true);
        // Descriptors formed once; a descriptor's start-address field holds
        // (address >> 4) and shared addresses stay below 256 KB, so an offset
        // within shared memory adds (offset >> 4).  Every instruction this
        // thread spends between MMAs costs tensor throughput (N=128 MMAs are
        // shorter than the issue path).
        const uint64_t q_desc = sw128_kmajor_desc(sb + P::Q_OFF);
        const uint64_t k_desc0 = sw128_kmajor_desc(sb + P::K_OFF);
        const uint64_t v_desc0 = sw128_mnmajor_desc(sb + P::V_OFF, P::BLK);
        const uint64_t qt_desc = sw32_desc(sb + P::Q_OFF + NB * P::BLK);
        const uint64_t kt_desc0 = sw32_desc(sb + P::K_OFF + NB * P::BLK);
        const uint64_t vt_desc0 = sw32_desc(sb + P::V_OFF + NB * P::BLK);
        bool ok = mbar_wait(q_full, 0, abort_flag);
        auto issue_s = [&](int j) -> bool {
            const int st = j % NS;                 // K stage
            const uint32_t ph = (j / NS) & 1;
            const int sbuf = j % P::SBUF;          // S buffer
            // S_j overwrites the columns of S_{j-2} / P_{j-2}: the softmax
            // finished with them before p_full(j-2), and PV_{j-2}, issued
            // earlier by this thread, reads P_{j-2} before this MMA writes
            // (MMAs of one thread execute in issue order)
            if (!mbar_wait(kv_full + 8 * st, ph, abort_flag)) return false;
            tc_fence_after();
            const uint32_t d = tmem + sbuf * TK;
            const uint32_t so = (st * P::TILE) >> 4;
#pragma unroll
            for (int kk = 0; kk < NB * 4; ++kk) {
                const uint32_t off = ((kk >> 2) * P::BLK + (kk & 3) * 32) >> 4;
                tc_mma_f16(d, q_desc + off, k_desc0 + so + off, idesc_s, kk > 0);
            }
            if constexpr (TAIL) tc_mma_f16(d, qt_desc, kt_desc0 + so, idesc_s, 1u);
            tc_commit(s_full + 8 * sbuf);
            tc_commit(k_empty + 8 * st);
            return true;
        };
        auto issue_pv = [&](int j) -> bool {
            const int st = j % NS;                 // V stage: landed with K_j (waited in issue_s)
            const int sbuf = j % P::SBUF;          // P lives in S buffer sbuf
            if (!mbar_wait(p_full, j & 1, abort_flag)) return false;
            tc_fence_after();
            const uint32_t so = (st * P::TILE) >> 4;
#pragma unroll
            for (int kk = 0; kk < TK / 16; ++kk) {
                const uint32_t a = tmem + sbuf * TK + kk * 8;    // P_j: 16 keys = 8 columns
                const uint32_t acc = (j > 0 || kk > 0) ? 1u : 0u;
                tc_mma_f16_ts(tmem + P::O_COL, a, v_desc0 + so + ((kk * 2048) >> 4), idesc_o, acc);
                if constexpr (TAIL)
                    tc_mma_f16_ts(tmem + P::O_COL + NB * 64, a, vt_desc0 + so + ((kk * 512) >> 4), idesc_ot,
                                  acc);
            }
            tc_commit(pv_done);
            tc_commit(v_empty + 8 * st);
            return true;
        };
        if (ok) ok = issue_s(0);
        // two S buffers: S_{j+1} runs while the softmax works on S_j; one
        // (DUO): S_{j+1} follows PV_j, which reads P_j from the same columns
        // (MMAs of one thread execute in issue order)
        for (int j = 1; ok && j < ntiles; ++j) ok = DUO ? (issue_pv(j - 1) && issue_s(j)) : (issue_s(j) && issue_pv(j - 1));
        if (ok) ok = issue_pv(ntiles - 1);
        if (!ok) fail();
        if (*abort_flag) {
            tc_commit(drain);
            mbar_wait(drain, 0, nullptr);
        }
    } else if (warp >= 2) {
        // ---------------- softmax: thread = query row
        const int q = warp & 3;
        const int row = q * 32 + lane;
        const uint32_t tl = tmem + (static_cast<uint32_t>(q * 32) << 16);
        float m_ref = -INFINITY, l = 0.f;
        bool ok = true;
        for (int j = 0; j < ntiles; ++j) {
            const int st = j % P::SBUF;
            const uint32_t ph = (j / P::SBUF) & 1;
            bool got = mbar_wait(s_full + 8 * st, ph, abort_flag);
            got = __all_sync(0xFFFFFFFFu, got);
            if (!got) { ok = false; break; }
            tc_fence_after();
            // all of S_j's loads in flight before one wait (the first wait
            // covers every load; the others tie each array to it)
            uint32_t r[TK / 32][32];
#pragma unroll
            for (int c = 0; c < TK / 32; ++c) tmem_ld_32x32b_x32(tl + st * TK + c * 32, r[c]);
#pragma unroll
            for (int c = 0; c < TK / 32; ++c) tmem_wait_ld_r(r[c]);
            float v[TK];
#pragma unroll
            for (int c = 0; c < TK / 32; ++c)
#pragma unroll
                for (int i = 0; i < 32; ++i) v[c * 32 + i] = __uint_as_float(r[c][i]);
            // raw scores: the row max is taken before scaling (scale > 0), and
            // keys past nk exist only in the last tile
            const int kvalid = nk - j * TK;
            if (kvalid < TK) {
#pragma unroll
                for (int i = 0; i < TK; ++i)
                    if (i >= kvalid) v[i] = -INFINITY;
            }
            // 8 independent max / sum chains (ILP instead of one 128-long chain)
            float mp[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) mp[u] = v[u];
#pragma unroll
            for (int i = 8; i < TK; ++i) mp[i & 7] = fmaxf(mp[i & 7], v[i]);
            float mt = fmaxf(fmaxf(fmaxf(mp[0], mp[1]), fmaxf(mp[2], mp[3])),
                             fmaxf(fmaxf(mp[4], mp[5]), fmaxf(mp[6], mp[7])));
            mt *= scale_log2;
            const bool resc = mt > m_ref + 8.f;
            const float m_new = resc ? mt : m_ref;
            const float corr = resc ? ex2_approx(m_ref - m_new) : 1.f;
            const float neg = -m_new;
            float sp[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int i = 0; i < TK; ++i) {
                v[i] = ex2_approx(fmaf(v[i], scale_log2, neg));
                sp[i & 7] += v[i];
            }
            const float rs = ((sp[0] + sp[1]) + (sp[2] + sp[3])) + ((sp[4] + sp[5]) + (sp[6] + sp[7]));
            l = l * corr + rs;
            m_ref = m_new;
            // P_j (bf16 pairs) over the first 64 columns of its own S buffer
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                uint32_t w[32];
#pragma unroll
                for (int i = 0; i < 32; ++i) w[i] = pack_bf16x2(v[64 * c + 2 * i], v[64 * c + 2 * i + 1]);
                tmem_st_32x32b_x32(tl + st * TK + c * 32, w);
            }
            tmem_wait_st();
            // PV_{j-1} must be done before O is rescaled; every phase is waited
            // so the parity stays in step with the barrier
            if (j > 0) {
                got = mbar_wait(pv_done, (j - 1) & 1, abort_flag);
                got = __all_sync(0xFFFFFFFFu, got);
                if (!got) { ok = false; break; }
                tc_fence_after();
            }
            if (j > 0 && __any_sync(0xFFFFFFFFu, resc)) {
#pragma unroll 1
                for (int c = 0; c < (HDP + 31) / 32; ++c) {
                    uint32_t r[32];
                    tmem_ld_32x32b_x32(tl + P::O_COL + c * 32, r);
                    tmem_wait_ld_r(r);
#pragma unroll
                    for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * corr);
                    tmem_st_32x32b_x32(tl + P::O_COL + c * 32, r);
                }
                tmem_wait_st();
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(p_full);
        }
        if (ok) {
            bool got = mbar_wait(pv_done, (ntiles - 1) & 1, abort_flag);
            got = __all_sync(0xFFFFFFFFu, got);
            ok = got;
        }
        if (!ok) {
            if (lane == 0) fail();
        } else {
            tc_fence_after();
            const float inv = 1.f / l;
            const int grow = qt * TQ + row;
            __nv_bfloat16* orow = O + (static_cast<size_t>(b) * nq + grow) * ldo + h * hd;
#pragma unroll 1
            for (int c = 0; c < (HDP + 31) / 32; ++c) {
                uint32_t r[32];
                tmem_ld_32x32b_x32(tl + P::O_COL + c * 32, r);
                tmem_wait_ld_r(r);
                if (grow < nq) {
#pragma unroll
                    for (int k4 = 0; k4 < 4; ++k4) {
                        if (c * 32 + 8 * k4 < hd) {
                            uint4 w;
                            w.x = pack_bf16x2(__uint_as_float(r[8 * k4 + 0]) * inv, __uint_as_float(r[8 * k4 + 1]) * inv);
                            w.y = pack_bf16x2(__uint_as_float(r[8 * k4 + 2]) * inv, __uint_as_float(r[8 * k4 + 3]) * inv);
                            w.z = pack_bf16x2(__uint_as_float(r[8 * k4 + 4]) * inv, __uint_as_float(r[8 * k4 + 5]) * inv);
                            w.w = pack_bf16x2(__uint_as_float(r[8 * k4 + 6]) * inv, __uint_as_float(r[8 * k4 + 7]) * inv);
                            *reinterpret_cast<uint4*>(orow + c * 32 + 8 * k4) = w;
                        }
                    }
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, P::TMEM_COLS);
    }
}

// [batch, rows, heads, hd] view of a bf16 matrix whose batch b, row r, head h
// starts at base + (b * rows + r) * ld + h * hd; box of box_cols x 1 head x
// 128 rows, columns past hd zero-filled.
bool make_map4(CUtensorMap* m, const void* base, int batch, int rows, int heads, int hd, int ld,
               int box_cols, CUtensorMapSwizzle sw) {
    EncodeTiledFn enc = tensor_map_encoder();
    if (!enc) return false;
    cuuint64_t dims[4] = {static_cast<cuuint64_t>(hd), static_cast<cuuint64_t>(heads),
                          static_cast<cuuint64_t>(rows), static_cast<cuuint64_t>(batch)};
    cuuint64_t strides[3] = {static_cast<cuuint64_t>(hd) * 2, static_cast<cuuint64_t>(ld) * 2,
                             static_cast<cuuint64_t>(ld) * 2 * static_cast<cuuint64_t>(rows)};
    cuuint32_t box[4] = {static_cast<cuuint32_t>(box_cols), 1, 128, 1};
    cuuint32_t es[4] = {1, 1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box,
               es, CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int NB, bool TAIL, bool DUO>
cudaError_t run_tc(const void* Q, const void* K, const void* V, void* O, int batch, int heads,
                   int hd, int nq, int nk, int ldq, int ldk, int ldv, int ldo, int* err,
                   cudaStream_t s, unsigned long long* launches) {
    using P = AttnPlan<NB, TAIL, DUO>;
    static_assert(P::BYTES <= 227 * 1024, "attention shared memory plan exceeds 227 KB");
    static bool attr = false;
    if (!attr) {
        cudaError_t e = cudaFuncSetAttribute(attn_tc_kernel<NB, TAIL, DUO>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, P::BYTES);
        if (e != cudaSuccess) return e;
        attr = true;
    }
    AttnMaps maps;
    const CUtensorMapSwizzle w128 = CU_TENSOR_MAP_SWIZZLE_128B, w32 = CU_TENSOR_MAP_SWIZZLE_32B;
    if (!make_map4(&maps.q, Q, batch, nq, heads, hd, ldq, 64, w128) ||
        !make_map4(&maps.k, K, batch, nk, heads, hd, ldk, 64, w128) ||
        !make_map4(&maps.v, V, batch, nk, heads, hd, ldv, 64, w128))
        return cudaErrorInvalidValue;
    if (TAIL) {
        if (!make_map4(&maps.qt, Q, batch, nq, heads, hd, ldq, 16, w32) ||
            !make_map4(&maps.kt, K, batch, nk, heads, hd, ldk, 16, w32) ||
            !make_map4(&maps.vt, V, batch, nk, heads, hd, ldv, 16, w32))
            return cudaErrorInvalidValue;
    } else {
        maps.qt = maps.q;
        maps.kt = maps.k;
        maps.vt = maps.v;
    }
    const float scale_log2 = 1.4426950408889634f / sqrtf(static_cast<float>(hd));
    dim3 grid((nq + TQ - 1) / TQ, heads, batch);
    cudaError_t le_ = launch_k(attn_tc_kernel<NB, TAIL, DUO>, grid, kThreadsA, P::BYTES, s, maps, static_cast<__nv_bfloat16*>(O), hd, nq, nk, ldo, scale_log2, err);
    ++*launches;
    return le_ != cudaSuccess ? le_ : cudaGetLastError();
}

// DLO_ATTN_DUO=0 keeps head dims up to 80 on one CTA per SM (tuning).
bool attn_duo_enabled() {
    static int v = -1;
    if (v < 0) {
        const char* e = std::getenv("DLO_ATTN_DUO");
        v = (e && e[0] == '0') ? 0 : 1;
    }
    return v != 0;
}

}  // namespace

bool attention_tc_supported(int hd) { return hd >= 8 && hd <= 128 && hd % 8 == 0; }

cudaError_t launch_attention_tc(const void* Q, const void* K, const void* V, void* O, int batch,
                                int heads, int hd, int nq, int nk, int ldq, int ldk, int ldv,
                                int ldo, int* err, cudaStream_t s, unsigned long long* launches) {
    // DUO when one CTA per SM would take more than one wave: with fewer CTAs
    // than SMs nothing shares an SM and the serial S / softmax / PV order of
    // a DUO CTA only costs time
    const long long ctas = static_cast<long long>((nq + TQ - 1) / TQ) * heads * batch;
    const bool duo = attn_duo_enabled() && ctas > gemm_num_sms();
    if (!attention_tc_supported(hd)) return cudaErrorInvalidValue;
    if (hd <= 64)
        return duo ? run_tc<1, false, true>(Q, K, V, O, batch, heads, hd, nq, nk, ldq, ldk, ldv, ldo, err, s, launches)
                   : run_tc<1, false, false>(Q, K, V, O, batch, heads, hd, nq, nk, ldq, ldk, ldv, ldo, err, s, launches);
    if (hd <= 80)
        return duo ? run_tc<1, true, true>(Q, K, V, O, batch, heads, hd, nq, nk, ldq, ldk, ldv, ldo, err, s, launches)
                   : run_tc<1, true, false>(Q, K, V, O, batch, heads, hd, nq, nk, ldq, ldk, ldv, ldo, err, s, launches);
    return run_tc<2, false, false>(Q, K, V, O, batch, heads, hd, nq, nk, ldq, ldk, ldv, ldo, err, s, launches);
}

cudaError_t launch_attention(const void* Q, const void* K, const void* V, void* O, int batch,
                             int heads, int hd, int nq, int nk, int ldq, int ldk, int ldv, int ldo,
                             int* err, cudaStream_t s, unsigned long long* launches) {
    if (nq <= 0 || batch <= 0 || heads <= 0) return cudaSuccess;
    if (nk <= 0) return cudaErrorInvalidValue;
    return launch_attention_tc(Q, K, V, O, batch, heads, hd, nq, nk, ldq, ldk, ldv, ldo, err, s, launches);
}

}  // namespace dlo
