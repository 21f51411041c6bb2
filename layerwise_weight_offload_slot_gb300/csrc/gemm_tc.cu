// Y = A W^T on the 5th-generation tensor cores (tcgen05), sm_103a.
//
// Persistent kernel, one CTA per SM, 6 warps (+12 converter warps for E4M3):
//   warp 0      TMA producer: 128x64 A tile and BNx64 W tile per stage (two
//               of each for 128-K stages), 128-byte swizzle, into a
//               STAGES-deep shared-memory ring
//   warp 1      TMEM owner and MMA issuer: tcgen05.mma kind::f16 (M=128,
//               N=BN, K=16) x 4 per stage into one of two fp32 TMEM
//               accumulators; tcgen05.commit frees the stage / publishes the
//               accumulator
//   warps 2..5  epilogue: warp q owns accumulator rows 32q..32q+31; per
//               column chunk it loads TMEM (tcgen05.ld), applies the
//               per-tensor scale, bias, GELU or gate, writes a 32-row box
//               into a 128-byte-swizzled shared-memory staging buffer and
//               lets TMA store it (bf16 outputs) or add it into the fp32
//               hidden state (cp.reduce.async.bulk .add: x += gate*(y + b)
//               without reading x).  Two staging buffers per warp let the
//               next chunk overlap the previous store.
// The two accumulators let the epilogue of tile t overlap the mainloop of
// tile t+1.  With E4M3 weights (FP8 = true) TMA loads the raw codes, twelve
// more warps widen them to bf16 in the swizzled layout the MMA reads (exact),
// and the per-tensor scale is applied to the fp32 accumulator in the epilogue.
// The widened tiles live in CB buffers of their own (conv / conv_empty
// barriers), so the ring of A tiles and raw codes is four stages deep.
// CTA pairs (gemm_pair_kernel, tcgen05 cta_group::2, below) take E4M3-weight
// GEMMs with at least 256 rows, and bf16 and W8A8 GEMMs where the tile model
// (pick_tile) finds them faster: one 256 x BN MMA over two SMs, each SM
// loading half of the weight tile.  W8A16 linears with many rows are widened
// to bf16 once, inside the pair kernel before its mainloop (WIDEN).
//
// Every mbarrier wait is bounded (2 s); a wait that runs out sets the
// kernel's error word and a CTA-wide abort flag, after which every role
// leaves its loop, in-flight TMA loads are drained (bounded) and TMEM is
// freed before exit.
#include <cuda.h>
#include <cuda_bf16.h>

#include <atomic>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <string>
#include <unordered_map>

#include "internal.h"
#include "ptx.cuh"

namespace dlo {

namespace {

constexpr int BM = 128;
constexpr int BK = 64;             // 64 bf16 = 128 bytes = one swizzle row
constexpr int A_TILE = BM * BK * 2;
constexpr int kThreads = 192;
constexpr int kConvWarps = 12;
constexpr int STG_BYTES = 32 * 128;   // one 32-row x 128-byte staging box

struct EpiArgs {
    int M, N, K;
    int epi;
    const __nv_bfloat16* bias;
    const float* scales;
    int scale_seg;
    const float* act_scale;   // W8A8: per-tensor activation scale (device), else NULL
    const float* gate;
    int gate_ld;
    int rows_per_batch;
    int* err;
    int num_m, num_n, num_tiles;
    int n_major;   // tile order: groups of N blocks sweep all M blocks (else the reverse)
    int group;     // blocks per group of the sweep (sweep_plan)
    int w_ready;   // W is not the preceding kernel's output (see GemmParams::w_ready)
    // W8A16 widened inside the pair kernel: E4M3 codes [N, K], the bf16
    // buffer the weight map reads, 16-code chunks, and the grid barrier's
    // counter (zero at launch)
    const uint4* wcodes;
    uint4* wwide;
    size_t wn16;
    unsigned* gbar;
};

// Grouped tile order: groups of `group` M-blocks sweep all N-blocks, so one
// group's A rows stay in L2 while the weights stream -- or, with n_major,
// groups of N-blocks sweep all M-blocks so the weight panel stays while A
// streams.  The host picks the order and group size (sweep_plan).
__device__ __forceinline__ void tile_coords(int t, const EpiArgs& a, int& mb, int& nb) {
    const int G = a.group;
    const int outer = a.n_major ? a.num_n : a.num_m, inner = a.n_major ? a.num_m : a.num_n;
    const int per_group = G * inner;
    const int g = t / per_group;
    const int first = g * G;
    const int gsz = min(outer - first, G);
    const int r = t - g * per_group;
    const int o = first + r % gsz, i = r / gsz;
    mb = a.n_major ? i : o;
    nb = a.n_major ? o : i;
}

// GELU, tanh approximation; tanh from the hardware approximation
// (relative error about 2^-11, below the bf16 rounding of the output).
__device__ __forceinline__ float gelu_tanh(float x) {
    const float k0 = 0.7978845608028654f, k1 = 0.044715f;
    return 0.5f * x * (1.f + tanh_approx(k0 * (x + k1 * x * x * x)));
}

// Byte offset of 16-byte chunk j of row r in a 128-byte-swizzled box.
__device__ __forceinline__ uint32_t sw128(int r, int j) {
    return static_cast<uint32_t>(r * 128 + ((j ^ (r & 7)) << 4));
}

// Scale (per 16-column segment) and bias of a 32-column chunk, loaded before
// the chunk's accumulator so their global-load latency overlaps the TMEM load.
struct EpiBS {
    float s[2];   // scale of each 16-column half
    uint4 b[4];   // bias, 8 bf16 per vector (zero without bias)
};

__device__ __forceinline__ void epi_load(const EpiArgs& a, float sa, int col0, EpiBS& e) {
#pragma unroll
    for (int g = 0; g < 2; ++g) {
        const int c = col0 + 16 * g;
        e.s[g] = a.scales ? (c < a.N ? a.scales[c / a.scale_seg] * sa : 0.f) : 1.f;
    }
#pragma unroll
    for (int q = 0; q < 4; ++q)
        e.b[q] = (a.bias && col0 + 8 * q < a.N) ? *reinterpret_cast<const uint4*>(a.bias + col0 + 8 * q)
                                                 : make_uint4(0, 0, 0, 0);
}

__device__ __forceinline__ void epi_apply(const EpiBS& e, float (&v)[32]) {
#pragma unroll
    for (int g = 0; g < 2; ++g)
#pragma unroll
        for (int i = 0; i < 16; ++i) v[16 * g + i] *= e.s[g];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const __nv_bfloat162* b2 = reinterpret_cast<const __nv_bfloat162*>(&e.b[q]);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float2 f = __bfloat1622float2(b2[j]);
            v[q * 8 + 2 * j] += f.x;
            v[q * 8 + 2 * j + 1] += f.y;
        }
    }
}

// e4m3 -> bf16, eight codes at a time, exactly.  For each code the 7
// exponent/mantissa bits go to bf16 bits 4..10 and the sign to bit 15, which
// is the same number scaled by 2^-120 (bf16 subnormals included); one bf16x2
// multiply by 2^120 restores it.  The magnitude bytes and the sign bits
// (pre-shifted to bit 3 of each byte) are interleaved into 16-bit lanes by
// one byte permute per pair of codes, and one shift by 4 places both.
// o[k] receives codes 2k and 2k+1 (code 0 = lowest byte of x0).
__device__ __forceinline__ void e4m3x8_to_bf16x8(uint32_t x0, uint32_t x1, uint32_t (&o)[4]) {
    constexpr uint32_t kScale = 0x7B807B80u;   // bf16x2 (2^120, 2^120)
    const uint32_t m0 = x0 & 0x7F7F7F7Fu, m1 = x1 & 0x7F7F7F7Fu;
    const uint32_t s0 = (x0 >> 4) & 0x08080808u, s1 = (x1 >> 4) & 0x08080808u;
    uint32_t w[4];
    asm("prmt.b32 %0, %1, %2, 0x5140;" : "=r"(w[0]) : "r"(m0), "r"(s0));
    asm("prmt.b32 %0, %1, %2, 0x7362;" : "=r"(w[1]) : "r"(m0), "r"(s0));
    asm("prmt.b32 %0, %1, %2, 0x5140;" : "=r"(w[2]) : "r"(m1), "r"(s1));
    asm("prmt.b32 %0, %1, %2, 0x7362;" : "=r"(w[3]) : "r"(m1), "r"(s1));
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const uint32_t t = w[k] << 4;
        asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(o[k]) : "r"(t), "r"(kScale));
    }
}

// E4M3 codes -> bf16, 16 codes per step and four steps in flight per thread
// (HBM-bound: 1 byte read, 2 written per weight); the last n % 16 codes
// (tail) by the first threads of block 0.
__global__ void __launch_bounds__(256) widen_e4m3_kernel(const uint4* __restrict__ codes,
                                                         uint4* __restrict__ out, size_t n16,
                                                         const uint8_t* __restrict__ tail_src,
                                                         uint16_t* __restrict__ tail_dst, int tail) {
    // the buffer written here may still be read by the preceding GEMM
    pdl_wait();
    pdl_launch_dependents();
    const size_t stride = static_cast<size_t>(gridDim.x) * blockDim.x;
    size_t i = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    auto widen16 = [&](size_t k, const uint4& v) {
        uint32_t lo[4], hi[4];
        e4m3x8_to_bf16x8(v.x, v.y, lo);
        e4m3x8_to_bf16x8(v.z, v.w, hi);
        out[2 * k] = make_uint4(lo[0], lo[1], lo[2], lo[3]);
        out[2 * k + 1] = make_uint4(hi[0], hi[1], hi[2], hi[3]);
    };
    for (; i + 3 * stride < n16; i += 4 * stride) {
        uint4 v[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) v[j] = __ldg(codes + i + j * stride);
#pragma unroll
        for (int j = 0; j < 4; ++j) widen16(i + j * stride, v[j]);
    }
    for (; i < n16; i += stride) widen16(i, __ldg(codes + i));
    if (blockIdx.x == 0 && static_cast<int>(threadIdx.x) < tail) {
        uint32_t o[4];
        e4m3x8_to_bf16x8(tail_src[threadIdx.x], 0u, o);
        tail_dst[threadIdx.x] = static_cast<uint16_t>(o[0] & 0xFFFFu);
    }
}

template <int BN, int STAGES, bool FP8, int MT = 1, int CB = 0, int KB = 1>
struct SmemPlan {
    // KB 64-wide K boxes per operand per stage (bf16: 128-K stages when 2)
    static constexpr int A_STAGE = MT * KB * A_TILE;      // MT x KB 128-row A boxes per stage
    static constexpr int W_BOX = BN * BK * 2;             // one bf16 weight box
    static constexpr int B_TILE = KB * W_BOX;             // bf16 operand tile (MMA reads)
    static constexpr int RAW_TILE = FP8 ? BN * BK : 0;     // e4m3 tile as loaded by TMA
    // bf16 B buffers: one per stage, or (E4M3, CB > 0) CB widened tiles that
    // cycle on their own, so the A / raw-code ring can be deeper than the
    // shared memory for a widened tile per stage would allow
    static constexpr int NBUF = (FP8 && CB) ? CB : STAGES;
    static constexpr int A_OFF = 0;
    static constexpr int B_OFF = STAGES * A_STAGE;
    static constexpr int RAW_OFF = B_OFF + NBUF * B_TILE;
    static constexpr int STG_OFF = RAW_OFF + STAGES * RAW_TILE;   // 4 warps x 2 boxes
    static constexpr int BAR_OFF = STG_OFF + 8 * STG_BYTES;
    // full[STAGES], empty[STAGES], conv[NBUF], conv_empty[NBUF], tfull[2], tempty[2], drain
    static constexpr int TMEM_SLOT_OFF = BAR_OFF + (2 * STAGES + 2 * NBUF + 5) * 8;
    static constexpr int ABORT_OFF = TMEM_SLOT_OFF + 4;
    static constexpr int BYTES = ABORT_OFF + 4 + 1024;  // + alignment slack
    static constexpr int THREADS = kThreads + (FP8 ? kConvWarps * 32 : 0);
    static constexpr uint32_t TX = A_STAGE + (FP8 ? RAW_TILE : B_TILE);
    // two accumulator sets of MT x BN fp32 columns; allocated in powers of two
    static constexpr uint32_t TMEM_COLS = 2 * MT * BN <= 256 ? 256u : 512u;
    static_assert(2 * MT * BN <= 512, "accumulators exceed TMEM");
    static_assert(KB == 1 || (!FP8 && CB == 0), "two K boxes per stage: bf16 operands");
};

// MT > 1: a CTA tile is MT x 128 rows; every weight tile (and, for E4M3,
// its widening) serves MT row blocks.  A8: A and W are both E4M3 codes
// (W8A8), multiplied by kind::f8f6f4 at 128 K per stage (the same 128-byte
// swizzled rows as bf16 at 64 K); no widening.
template <int BN, int STAGES, bool FP8, int MT, bool A8, int CB = 0, int KB = 1>
__global__ void __launch_bounds__(SmemPlan<BN, STAGES, FP8, MT, CB, KB>::THREADS, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                const __grid_constant__ CUtensorMap tmO, const EpiArgs args) {
    static_assert(!(A8 && FP8), "W8A8 loads 8-bit codes for both operands, nothing to widen");
    static_assert(KB == 1 || !A8, "W8A8 stages are one 128-byte box wide");
    using P = SmemPlan<BN, STAGES, FP8, MT, CB, KB>;
    constexpr bool DEC = FP8 && CB > 0;   // widened tiles decoupled from the stages
    // K elements per stage: 128 bytes of a row per box either way
    constexpr int KS = A8 ? 128 : BK * KB;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const uint32_t sbase = smem_u32(smem);
    const uint32_t bar_full = sbase + P::BAR_OFF;
    const uint32_t bar_empty = bar_full + STAGES * 8;
    const uint32_t bar_conv = bar_empty + STAGES * 8;
    const uint32_t bar_cempty = bar_conv + P::NBUF * 8;
    const uint32_t bar_tfull = bar_cempty + P::NBUF * 8;
    const uint32_t bar_tempty = bar_tfull + 2 * 8;
    const uint32_t bar_drain = bar_tempty + 2 * 8;
    volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(smem + P::TMEM_SLOT_OFF);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + P::ABORT_OFF);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(bar_full + s * 8, 1);
            mbar_init(bar_empty + s * 8, 1);
        }
        for (int c = 0; c < P::NBUF; ++c) {
            mbar_init(bar_conv + c * 8, kConvWarps);
            mbar_init(bar_cempty + c * 8, 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(bar_tfull + a * 8, 1);
            mbar_init(bar_tempty + a * 8, 4);
        }
        mbar_init(bar_drain, 1);
        *abort_flag = 0;
        fence_mbar_init();
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
        tma_prefetch_desc(&tmO);
    }
    if (warp == 1) {
        tmem_alloc(sbase + P::TMEM_SLOT_OFF, P::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    const int kblocks = (args.K + KS - 1) / KS;
    // predecessor's outputs complete and visible; the producer waits after
    // its weight prefetch when the weights are not a predecessor's output
    const bool prefetch_w = args.w_ready && warp == 0 && lane == 0;
    if (!prefetch_w) {
        pdl_wait();
        pdl_launch_dependents();
    }

    auto fail = [&]() {
        *abort_flag = 1;
        if (args.err) atomicExch(args.err, 1);
    };

    if (warp == 0 && lane == 0) {
        // ---------------- TMA producer
        int s = 0;
        uint32_t ph = 0;
        bool ok = true;
        uint32_t issued = 0, last_par = 0;   // per-stage bit masks
        auto load_w = [&](int st, int kb, int nb) {
            if constexpr (FP8) {
                tma_load_2d(sbase + P::RAW_OFF + st * P::RAW_TILE, &tmB, kb * KS, nb * BN, bar_full + st * 8);
            } else {
#pragma unroll
                for (int b = 0; b < KB; ++b)
                    tma_load_2d(sbase + P::B_OFF + st * P::B_TILE + b * P::W_BOX, &tmB, kb * KS + b * BK, nb * BN,
                                bar_full + st * 8);
            }
        };
        // weight tiles of the first tile's first stages (the stages start
        // empty), before the programmatic-launch wait
        int pre = 0;
        if (prefetch_w) {
            if (static_cast<int>(blockIdx.x) < args.num_tiles) {
                int mb0, nb0;
                tile_coords(blockIdx.x, args, mb0, nb0);
                pre = kblocks < STAGES ? kblocks : STAGES;
                for (int st = 0; st < pre; ++st) {
                    mbar_arrive_expect_tx(bar_full + st * 8, P::TX);
                    load_w(st, st, nb0);
                    issued |= 1u << st;   // phase 0 (the drain on abort waits for it)
                }
            }
            pdl_wait();
            pdl_launch_dependents();
        }
        for (int tile = blockIdx.x; ok && tile < args.num_tiles; tile += gridDim.x) {
            int mb, nb;
            tile_coords(tile, args, mb, nb);
            for (int kb = 0; kb < kblocks; ++kb) {
                if (!mbar_wait(bar_empty + s * 8, ph ^ 1, abort_flag)) {
                    fail();
                    ok = false;
                    break;
                }
                const uint32_t fb = bar_full + s * 8;
                const bool w_done = tile == static_cast<int>(blockIdx.x) && kb < pre;
                if (!w_done) mbar_arrive_expect_tx(fb, P::TX);
#pragma unroll
                for (int i = 0; i < MT; ++i)
#pragma unroll
                    for (int b = 0; b < KB; ++b)
                        tma_load_2d(sbase + P::A_OFF + s * P::A_STAGE + (i * KB + b) * A_TILE, &tmA,
                                    kb * KS + b * BK, (mb * MT + i) * BM, fb);
                if (!w_done) load_w(s, kb, nb);
                issued |= 1u << s;
                last_par = (last_par & ~(1u << s)) | (ph << s);
                if (++s == STAGES) {
                    s = 0;
                    ph ^= 1;
                }
            }
        }
        if (!ok || *abort_flag) {
            // drain: the last load issued into each stage must land before
            // the CTA exits (bounded wait on that fill's phase)
            for (int i = 0; i < STAGES; ++i)
                if (issued & (1u << i)) mbar_wait(bar_full + i * 8, (last_par >> i) & 1u, nullptr);
        }
    } else if (warp == 1 && lane == 0) {
        // ---------------- MMA issuer
        constexpr uint32_t idesc = A8 ? idesc_e4m3_f32(BM, BN) : idesc_bf16_f32(BM, BN);
        const uint32_t bar_ready = FP8 ? bar_conv : bar_full;
        // Operand descriptors are formed once: a descriptor's start-address
        // field holds (address >> 4) and shared addresses stay below 256 KB,
        // so moving within shared memory adds (offset >> 4).  The issuing
        // thread's instructions between MMAs cost tensor throughput for
        // MMAs shorter than the issue path (N <= 192), so the stage loop
        // only adds constants.
        const uint64_t a_desc0 = sw128_kmajor_desc(sbase + P::A_OFF);
        const uint64_t b_desc0 = sw128_kmajor_desc(sbase + P::B_OFF);
        uint64_t a_desc = a_desc0, b_desc = b_desc0;
        int s = 0;
        uint32_t ph = 0;
        int cb = 0;          // DEC: widened buffer and its phase
        uint32_t cph = 0;
        int t = 0;
        bool ok = true;
        for (int tile = blockIdx.x; ok && tile < args.num_tiles; tile += gridDim.x, ++t) {
            const int acc = t & 1;
            const uint32_t aph = (t >> 1) & 1;
            if (!mbar_wait(bar_tempty + acc * 8, aph ^ 1, abort_flag)) {
                fail();
                break;
            }
            tc_fence_after();
            const uint32_t d_tmem = tmem_base + acc * (MT * BN);
            for (int kb = 0; kb < kblocks; ++kb) {
                if (!mbar_wait(DEC ? bar_conv + cb * 8 : bar_ready + s * 8, DEC ? cph : ph, abort_flag)) {
                    fail();
                    ok = false;
                    break;
                }
                tc_fence_after();
#pragma unroll
                for (int i = 0; i < MT; ++i) {
#pragma unroll
                    for (int b = 0; b < KB; ++b) {
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk) {   // 4 x 32 bytes of K per box
                            const uint64_t ad = a_desc + (((i * KB + b) * A_TILE + kk * 32) >> 4);
                            const uint64_t bd = b_desc + ((b * P::W_BOX + kk * 32) >> 4);
                            if constexpr (A8)
                                tc_mma_f8(d_tmem + i * BN, ad, bd, idesc, (kb | kk) != 0);
                            else
                                tc_mma_f16(d_tmem + i * BN, ad, bd, idesc, (kb | b | kk) != 0);
                        }
                    }
                }
                tc_commit(bar_empty + s * 8);
                if constexpr (DEC) {
                    tc_commit(bar_cempty + cb * 8);
                    if (++cb == P::NBUF) {
                        cb = 0;
                        cph ^= 1;
                        b_desc = b_desc0;
                    } else {
                        b_desc += P::B_TILE >> 4;
                    }
                    if (++s == STAGES) {
                        s = 0;
                        ph ^= 1;
                        a_desc = a_desc0;
                    } else {
                        a_desc += P::A_STAGE >> 4;
                    }
                } else if (++s == STAGES) {
                    s = 0;
                    ph ^= 1;
                    a_desc = a_desc0;
                    b_desc = b_desc0;
                } else {
                    a_desc += P::A_STAGE >> 4;
                    b_desc += P::B_TILE >> 4;
                }
            }
            if (ok) tc_commit(bar_tfull + acc * 8);
        }
        if (*abort_flag) {
            // drain: wait (bounded) until every MMA issued so far completed
            tc_commit(bar_drain);
            mbar_wait(bar_drain, 0, nullptr);
        }
    } else if (warp >= 2 && warp < 6) {
        // ---------------- epilogue: warp q owns accumulator rows 32q .. 32q+31
        const int q = warp & 3;
        const uint32_t stg0 = sbase + P::STG_OFF + q * 2 * STG_BYTES;
        uint8_t* stg0p = smem + P::STG_OFF + q * 2 * STG_BYTES;
        int bi = 0;   // staging buffer toggle
        int t = 0;
        const bool residual = args.epi == DLO_EPI_RESIDUAL;
        for (int tile = blockIdx.x; tile < args.num_tiles; tile += gridDim.x, ++t) {
            const int acc = t & 1;
            const uint32_t aph = (t >> 1) & 1;
            int mb, nb;
            tile_coords(tile, args, mb, nb);
            const float sa = (args.scales && args.act_scale) ? *args.act_scale : 1.0f;
            bool ok = mbar_wait(bar_tfull + acc * 8, aph, abort_flag);
            ok = __all_sync(0xFFFFFFFFu, ok);
            if (!ok) {
                if (lane == 0) fail();
                break;
            }
            tc_fence_after();
#pragma unroll 1
            for (int mi = 0; mi < MT; ++mi) {
                const int row0 = (mb * MT + mi) * BM + q * 32;
                const int row = row0 + lane;
                const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                                       acc * (MT * BN) + mi * BN;
                if (residual) {
                    // 32-column fp32 boxes: delta = gate * (acc * s + b), added into x by TMA
                    const float* grow = args.gate ? args.gate + static_cast<size_t>(min(row, args.M - 1) /
                                                                                     args.rows_per_batch) *
                                                                    args.gate_ld
                                                  : nullptr;
    #pragma unroll 1
                    for (int c0 = 0; c0 < BN; c0 += 32) {
                        const int col0 = nb * BN + c0;
                        if (col0 >= args.N) break;
                        EpiBS e;
                        epi_load(args, sa, col0, e);
                        float4 gv[8];
    #pragma unroll
                        for (int j = 0; j < 8; ++j)
                            gv[j] = (grow && col0 + 4 * j < args.N)
                                        ? *reinterpret_cast<const float4*>(grow + col0 + 4 * j)
                                        : make_float4(1.f, 1.f, 1.f, 1.f);
                        uint32_t r[32];
                        tmem_ld_32x32b_x32_nc(taddr + c0, r);
                        tmem_wait_ld_r(r);
                        float v[32];
    #pragma unroll
                        for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
                        epi_apply(e, v);
    #pragma unroll
                        for (int j = 0; j < 8; ++j) {
                            v[4 * j] *= gv[j].x;
                            v[4 * j + 1] *= gv[j].y;
                            v[4 * j + 2] *= gv[j].z;
                            v[4 * j + 3] *= gv[j].w;
                        }
                        if (lane == 0) bulk_wait_read<1>();
                        __syncwarp();
                        uint8_t* box = stg0p + bi * STG_BYTES;
    #pragma unroll
                        for (int j = 0; j < 8; ++j)
                            *reinterpret_cast<float4*>(box + sw128(lane, j)) =
                                make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
                        fence_proxy_async_smem();
                        __syncwarp();
                        if (lane == 0) {
                            tma_reduce_add_2d(&tmO, stg0 + bi * STG_BYTES, col0, row0);
                            bulk_commit();
                        }
                        bi ^= 1;
                    }
                } else {
                    // 64-column bf16 boxes: y = [GELU](acc * s + b), stored by TMA;
                    // filled 32 columns at a time to keep registers low
    #pragma unroll 1
                    for (int c0 = 0; c0 < BN; c0 += 64) {
                        const int col0 = nb * BN + c0;
                        if (col0 >= args.N) break;
                        if (lane == 0) bulk_wait_read<1>();
                        __syncwarp();
                        uint8_t* box = stg0p + bi * STG_BYTES;
                        EpiBS e2[2];
                        epi_load(args, sa, col0, e2[0]);
                        epi_load(args, sa, col0 + 32, e2[1]);
    #pragma unroll
                        for (int half = 0; half < 2; ++half) {
                            uint32_t r[32];
                            tmem_ld_32x32b_x32_nc(taddr + c0 + 32 * half, r);
                            tmem_wait_ld_r(r);
                            float v[32];
    #pragma unroll
                            for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
                            epi_apply(e2[half], v);
                            if (args.epi == DLO_EPI_GELU) {
    #pragma unroll
                                for (int i = 0; i < 32; ++i) v[i] = gelu_tanh(v[i]);
                            }
    #pragma unroll
                            for (int j = 0; j < 4; ++j) {
                                uint4 w;
                                w.x = pack_bf16x2(v[8 * j + 0], v[8 * j + 1]);
                                w.y = pack_bf16x2(v[8 * j + 2], v[8 * j + 3]);
                                w.z = pack_bf16x2(v[8 * j + 4], v[8 * j + 5]);
                                w.w = pack_bf16x2(v[8 * j + 6], v[8 * j + 7]);
                                *reinterpret_cast<uint4*>(box + sw128(lane, 4 * half + j)) = w;
                            }
                        }
                        fence_proxy_async_smem();
                        __syncwarp();
                        if (lane == 0) {
                            tma_store_2d(&tmO, stg0 + bi * STG_BYTES, col0, row0);
                            bulk_commit();
                        }
                        bi ^= 1;
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_tempty + acc * 8);
        }
        if (lane == 0) bulk_wait_all();
        __syncwarp();
    } else if constexpr (FP8) {
        if (warp >= 6) {
            // ---------------- e4m3 -> bf16 converters (kConvWarps warps)
            const int ct = threadIdx.x - 6 * 32;
            int s = 0;
            uint32_t ph = 0;
            int cb = 0;
            uint32_t cph = 0;
            bool ok = true;
            for (int tile = blockIdx.x; ok && tile < args.num_tiles; tile += gridDim.x) {
                for (int kb = 0; kb < kblocks; ++kb) {
                    bool got = mbar_wait(bar_full + s * 8, ph, abort_flag);
                    if (DEC && got) got = mbar_wait(bar_cempty + cb * 8, cph ^ 1, abort_flag);
                    got = __all_sync(0xFFFFFFFFu, got);
                    if (!got) {
                        if (lane == 0) fail();
                        ok = false;
                        break;
                    }
                    const uint8_t* raw = smem + P::RAW_OFF + s * P::RAW_TILE;
                    uint8_t* dst = smem + P::B_OFF + (DEC ? cb : s) * P::B_TILE;
#pragma unroll 4
                    for (int i = ct; i < BN * 8; i += kConvWarps * 32) {
                        const int r = i >> 3, c = i & 7;
                        const uint2 v = *reinterpret_cast<const uint2*>(raw + r * 64 + c * 8);
                        uint32_t o[4];
                        e4m3x8_to_bf16x8(v.x, v.y, o);
                        *reinterpret_cast<uint4*>(dst + sw128(r, c)) = make_uint4(o[0], o[1], o[2], o[3]);
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bar_conv + (DEC ? cb : s) * 8);
                    if (++s == STAGES) {
                        s = 0;
                        ph ^= 1;
                    }
                    if (DEC && ++cb == P::NBUF) {
                        cb = 0;
                        cph ^= 1;
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
        tmem_dealloc(tmem_base, P::TMEM_COLS);
    }
}

// ------------------------------------------------------------------ CTA-pair GEMM
//
// GEMMs on CTA pairs (tcgen05 cta_group::2).  A cluster of two CTAs computes
// one 256 x BN output tile.  CTA r (its rank in the cluster) loads the tile's
// A rows 128r .. 128r+127 and the tile's weight rows BN/2*r .. BN/2*r+BN/2-1,
// and holds accumulator rows 128r .. 128r+127 (128 lanes x BN fp32 columns,
// two sets) in its own tensor memory.  Rank 0's MMA thread issues one
// M = 256, N = BN, K = 16 MMA per 32-byte K step for both CTAs once both
// halves of the stage are ready; the MMA commits reach both CTAs (multicast).
// Per SM a 64-K step is a 128 x BN x 64 product fed by 16 KB of A and only
// BN/2 weight rows: half the weight bytes per FLOP of a single-CTA tile of
// the same width, which matters because an SM takes in operand bytes from L2
// at ~70 bytes per cycle while all SMs stream.
//
// bf16 weights (FP8 = false): TMA loads both operands into a STAGES-deep
// ring.  E4M3 weights (FP8 = true, BN = 256): TMA loads the raw codes, twelve
// converter warps widen this CTA's weight rows into CB widened buffers of
// their own (as gemm_kernel's), and the per-tensor scale is applied in the
// epilogue.  W8A8 (A8): both operands are E4M3 codes in the same 128-byte
// rows (128 K per stage), multiplied by kind::f8f6f4 MMAs of K = 32; the
// epilogue applies the activation scale times the weight scale.
//
// Readiness of rank 1's half crosses to rank 0 once per step without a fence
// on any thread: rank 1's warp 1, idle otherwise, waits until the half is
// ready in its own CTA (its stage's TMA loads landed; with E4M3 also its
// converter warps' widened tile, ordered for the async proxy by
// fence.proxy.async) and then issues a 16-byte bulk copy into rank 0's
// shared memory whose completion lands as transaction bytes on the rank-0
// barrier the MMA thread waits on.  A cluster-scope release arrival would
// cost ~550 ns per step (measured), more than the step's MMAs.  Each CTA runs
// gemm_kernel's epilogue on its own 128 rows, then arrives on rank 0's
// accumulator-free barrier.
template <int BN, int STAGES, int CB, bool FP8, bool A8 = false>
struct PairPlan {
    static constexpr int KS = A8 ? 128 : BK;               // K elements per stage (128-byte rows)
    static constexpr int HALF = BN / 2;                    // weight rows each CTA loads
    static constexpr int BM2 = 2 * BM;                     // output rows of a pair tile
    static constexpr int NW = FP8 ? CB : STAGES;           // bf16 weight buffers the MMA reads
    static constexpr int NCB = FP8 ? CB : 0;               // widened-buffer barrier sets
    static constexpr int RAW_TILE = FP8 ? HALF * BK : 0;   // codes of one CTA's weight rows
    static constexpr int W_TILE = HALF * BK * 2;           // bf16 weight rows (MMA reads)
    static constexpr int A_OFF = 0;
    static constexpr int W_OFF = STAGES * A_TILE;
    static constexpr int RAW_OFF = W_OFF + NW * W_TILE;
    static constexpr int STG_OFF = RAW_OFF + STAGES * RAW_TILE;   // 4 warps x 2 boxes
    static constexpr int BAR_OFF = STG_OFF + 8 * STG_BYTES;
    // full[STAGES], empty[STAGES], (E4M3: conv[CB], cempty[CB], wdone[CB]),
    // tfull[2], tempty[2], drain, then a 16-byte slot the forwarded bulk
    // copies land in
    static constexpr int SIG_OFF = (BAR_OFF + (2 * STAGES + 3 * NCB + 5) * 8 + 15) / 16 * 16;
    static constexpr int TMEM_SLOT_OFF = SIG_OFF + 16;
    static constexpr uint32_t SIG_BYTES = 16;
    static constexpr int ABORT_OFF = TMEM_SLOT_OFF + 4;
    static constexpr int BYTES = ABORT_OFF + 4 + 1024;   // + alignment slack
    static constexpr int THREADS = kThreads + (FP8 ? kConvWarps * 32 : 0);
    static constexpr uint32_t TX = A_TILE + (FP8 ? RAW_TILE : W_TILE);
    // two accumulator sets of BN fp32 columns; allocated in powers of two
    static constexpr uint32_t TMEM_COLS = 2 * BN <= 256 ? 256u : 512u;
    static_assert(BN % 64 == 0 && BN >= 128 && BN <= 256, "pair tile width: 128, 192 or 256");
    static_assert(!FP8 || (BN == 256 && CB > 0), "E4M3 pairs: 256-wide tiles, widened buffers");
    static_assert(!(FP8 && A8), "W8A8 multiplies the codes, nothing to widen");
    static_assert(W_OFF % 1024 == 0 && RAW_OFF % 1024 == 0 && STG_OFF % 1024 == 0 && W_TILE % 1024 == 0,
                  "swizzled buffers must be 1024-B aligned");
};

template <int BN, int STAGES, int CB, bool FP8, bool A8 = false, bool WIDEN = false>
__global__ void __launch_bounds__(PairPlan<BN, STAGES, CB, FP8, A8>::THREADS, 1)
    gemm_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                     const __grid_constant__ CUtensorMap tmO, const EpiArgs args) {
    using P = PairPlan<BN, STAGES, CB, FP8, A8>;
    static_assert(!WIDEN || (!FP8 && !A8), "widening prologue: bf16 mainloop");
    constexpr int KS = P::KS;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const uint32_t sbase = smem_u32(smem);
    const uint32_t bar_full = sbase + P::BAR_OFF;
    const uint32_t bar_empty = bar_full + STAGES * 8;
    const uint32_t bar_conv = bar_empty + STAGES * 8;     // E4M3 only (NCB = 0 otherwise)
    const uint32_t bar_cempty = bar_conv + P::NCB * 8;
    const uint32_t bar_wdone = bar_cempty + P::NCB * 8;
    const uint32_t bar_tfull = bar_wdone + P::NCB * 8;
    const uint32_t bar_tempty = bar_tfull + 2 * 8;
    const uint32_t bar_drain = bar_tempty + 2 * 8;
    volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(smem + P::TMEM_SLOT_OFF);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + P::ABORT_OFF);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    // launched in anything but clusters of two (a tool replaying the launch
    // without its cluster shape, say), the pair instructions below would be
    // invalid: report it and do nothing
    if (cluster_nctarank() != 2) {
        if (threadIdx.x == 0 && args.err) atomicExch(args.err, 1);
        return;
    }
    const uint32_t rank = cluster_ctarank();
    const int pair = static_cast<int>(blockIdx.x >> 1), npairs = static_cast<int>(gridDim.x >> 1);

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(bar_full + s * 8, 1);
            mbar_init(bar_empty + s * 8, 1);
        }
        for (int c = 0; c < P::NCB; ++c) {
            // rank 0's converter warps (one of them also expects the bytes
            // rank 1 forwards)
            mbar_init(bar_conv + c * 8, kConvWarps);
            mbar_init(bar_cempty + c * 8, 1);
            mbar_init(bar_wdone + c * 8, kConvWarps);   // rank 1: its converter warps
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(bar_tfull + a * 8, 1);
            mbar_init(bar_tempty + a * 8, 8);              // both CTAs' epilogue warps
        }
        mbar_init(bar_drain, 1);
        *abort_flag = 0;
        fence_mbar_init();
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
        tma_prefetch_desc(&tmO);
    }
    if (warp == 1) {
        tmem_alloc_pair(sbase + P::TMEM_SLOT_OFF, P::TMEM_COLS);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    __syncthreads();
    // the peer's barriers are initialised before anything arrives on them
    cluster_sync_all();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    const int kblocks = (args.K + KS - 1) / KS;
    // the rank-0 barriers rank 1's readiness lands on (E4M3: the widened
    // buffers'; bf16: the stages'), its accumulator-free barriers and the
    // signal slot, as shared::cluster addresses
    const uint32_t ready_r0 = mapa_shared(FP8 ? bar_conv : bar_full, 0);
    const uint32_t tempty_r0 = mapa_shared(bar_tempty, 0);
    const uint32_t sig_r0 = mapa_shared(sbase + P::SIG_OFF, 0);
    // weights are never the predecessor's output (w_ready): the producer's
    // first weight tiles may load before the programmatic-launch wait
    const bool prefetch_w = args.w_ready && warp == 0 && lane == 0;
    if (!prefetch_w) {
        pdl_wait();
        pdl_launch_dependents();
    }

    auto fail = [&]() {
        *abort_flag = 1;
        if (args.err) atomicExch(args.err, 1);
    };

    if constexpr (WIDEN) {
        // ---------------- W8A16 inside the GEMM: every thread of the grid
        // widens a share of the linear's E4M3 codes into the bf16 buffer the
        // weight map reads (the predecessor, which may have read that buffer,
        // has completed: every thread passed the programmatic-launch wait),
        // then the grid meets at a barrier (cooperative launch: all CTAs
        // co-resident; bounded) before the first weight tile is loaded
        const size_t stride = static_cast<size_t>(gridDim.x) * blockDim.x;
        size_t i = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x;
        auto widen16 = [&](size_t k, const uint4& v) {
            uint32_t lo[4], hi[4];
            e4m3x8_to_bf16x8(v.x, v.y, lo);
            e4m3x8_to_bf16x8(v.z, v.w, hi);
            args.wwide[2 * k] = make_uint4(lo[0], lo[1], lo[2], lo[3]);
            args.wwide[2 * k + 1] = make_uint4(hi[0], hi[1], hi[2], hi[3]);
        };
        for (; i + 7 * stride < args.wn16; i += 8 * stride) {
            uint4 v[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) v[j] = __ldg(args.wcodes + i + j * stride);
#pragma unroll
            for (int j = 0; j < 8; ++j) widen16(i + j * stride, v[j]);
        }
        for (; i < args.wn16; i += stride) widen16(i, __ldg(args.wcodes + i));
        fence_proxy_async_global();
        __syncthreads();
        if (threadIdx.x == 0 && !grid_arrive_wait(args.gbar, gridDim.x, abort_flag)) fail();
        __syncthreads();
        fence_proxy_async_global();
    }

    if (warp == 0 && lane == 0) {
        // ---------------- TMA producer: this CTA's A rows and weight rows
        // (bf16: rank 0's stage also waits for rank 1's forwarded bytes)
        constexpr uint32_t tx0 = FP8 ? P::TX : P::TX + P::SIG_BYTES;
        const uint32_t tx = rank == 0 ? tx0 : P::TX;
        int s = 0;
        uint32_t ph = 0;
        bool ok = true;
        uint32_t issued = 0, last_par = 0;
        auto load_w = [&](int st, int kb, int nb) {
            const int wrow = nb * BN + static_cast<int>(rank) * P::HALF;
            if constexpr (FP8)
                tma_load_2d(sbase + P::RAW_OFF + st * P::RAW_TILE, &tmB, kb * KS, wrow, bar_full + st * 8);
            else
                tma_load_2d(sbase + P::W_OFF + st * P::W_TILE, &tmB, kb * KS, wrow, bar_full + st * 8);
        };
        int pre = 0;
        if (prefetch_w) {
            if (pair < args.num_tiles) {
                int mb0, nb0;
                tile_coords(pair, args, mb0, nb0);
                pre = kblocks < STAGES ? kblocks : STAGES;
                for (int st = 0; st < pre; ++st) {
                    mbar_arrive_expect_tx(bar_full + st * 8, tx);
                    load_w(st, st, nb0);
                    issued |= 1u << st;
                }
            }
            pdl_wait();
            pdl_launch_dependents();
        }
        for (int tile = pair; ok && tile < args.num_tiles; tile += npairs) {
            int mb, nb;
            tile_coords(tile, args, mb, nb);
            for (int kb = 0; kb < kblocks; ++kb) {
                if (!mbar_wait(bar_empty + s * 8, ph ^ 1, abort_flag)) {
                    fail();
                    ok = false;
                    break;
                }
                const uint32_t fb = bar_full + s * 8;
                const bool w_done = tile == pair && kb < pre;
                if (!w_done) mbar_arrive_expect_tx(fb, tx);
                tma_load_2d(sbase + P::A_OFF + s * A_TILE, &tmA, kb * KS,
                            mb * P::BM2 + static_cast<int>(rank) * BM, fb);
                if (!w_done) load_w(s, kb, nb);
                issued |= 1u << s;
                last_par = (last_par & ~(1u << s)) | (ph << s);
                if (++s == STAGES) {
                    s = 0;
                    ph ^= 1;
                }
            }
        }
        if (!ok || *abort_flag) {
            for (int i = 0; i < STAGES; ++i)
                if (issued & (1u << i)) mbar_wait(bar_full + i * 8, (last_par >> i) & 1u, nullptr);
        }
    } else if (warp == 1 && lane == 0 && rank == 0) {
        // ---------------- MMA issuer of the pair (rank 0 only)
        constexpr uint32_t idesc = A8 ? idesc_e4m3_f32(P::BM2, BN) : idesc_bf16_f32(P::BM2, BN);
        const uint64_t a_desc0 = sw128_kmajor_desc(sbase + P::A_OFF);
        const uint64_t b_desc0 = sw128_kmajor_desc(sbase + P::W_OFF);
        uint64_t a_desc = a_desc0, b_desc = b_desc0;
        int s = 0, cb = 0;
        uint32_t ph = 0, cph = 0;
        int t = 0;
        bool ok = true;
        for (int tile = pair; ok && tile < args.num_tiles; tile += npairs, ++t) {
            const int acc = t & 1;
            const uint32_t aph = (t >> 1) & 1;
            if (!mbar_wait_cluster(bar_tempty + acc * 8, aph ^ 1, abort_flag)) {
                fail();
                break;
            }
            tc_fence_after();
            const uint32_t d_tmem = tmem_base + acc * BN;
            for (int kb = 0; kb < kblocks; ++kb) {
                const bool got = FP8 ? mbar_wait_cluster(bar_conv + cb * 8, cph, abort_flag)
                                     : mbar_wait_cluster(bar_full + s * 8, ph, abort_flag);
                if (!got) {
                    fail();
                    ok = false;
                    break;
                }
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {   // 4 x 32 bytes of K per stage
                    if constexpr (A8)
                        tc_mma_f8_pair(d_tmem, a_desc + ((kk * 32) >> 4), b_desc + ((kk * 32) >> 4), idesc,
                                       (kb | kk) != 0);
                    else
                        tc_mma_f16_pair(d_tmem, a_desc + ((kk * 32) >> 4), b_desc + ((kk * 32) >> 4), idesc,
                                        (kb | kk) != 0);
                }
                tc_commit_pair_mc(bar_empty + s * 8, 3);
                if constexpr (FP8) {
                    tc_commit_pair_mc(bar_cempty + cb * 8, 3);
                    if (++cb == CB) {
                        cb = 0;
                        cph ^= 1;
                        b_desc = b_desc0;
                    } else {
                        b_desc += P::W_TILE >> 4;
                    }
                    if (++s == STAGES) {
                        s = 0;
                        ph ^= 1;
                        a_desc = a_desc0;
                    } else {
                        a_desc += A_TILE >> 4;
                    }
                } else if (++s == STAGES) {
                    s = 0;
                    ph ^= 1;
                    a_desc = a_desc0;
                    b_desc = b_desc0;
                } else {
                    a_desc += A_TILE >> 4;
                    b_desc += P::W_TILE >> 4;
                }
            }
            if (ok) tc_commit_pair_mc(bar_tfull + acc * 8, 3);
        }
        if (*abort_flag) {
            // drain: wait (bounded) until every MMA issued so far completed
            tc_commit_pair(bar_drain);
            mbar_wait(bar_drain, 0, nullptr);
        }
    } else if (warp == 1 && lane == 0) {
        // ---------------- rank 1: forward each ready half to rank 0
        // (E4M3: per widened buffer, after its converter warps; bf16: per
        // stage, after its TMA loads)
        constexpr int NR = FP8 ? CB : STAGES;
        const uint32_t ready_local = FP8 ? bar_wdone : bar_full;
        int r = 0;
        uint32_t rph = 0;
        bool ok = true;
        for (int tile = pair; ok && tile < args.num_tiles; tile += npairs) {
            for (int kb = 0; kb < kblocks; ++kb) {
                if (!mbar_wait(ready_local + r * 8, rph, abort_flag)) {
                    fail();
                    ok = false;
                    break;
                }
                fence_proxy_async_smem();
                bulk_s2s_cluster(sig_r0, sbase + P::SIG_OFF, P::SIG_BYTES, ready_r0 + r * 8);
                if (++r == NR) {
                    r = 0;
                    rph ^= 1;
                }
            }
        }
    } else if (warp >= 2 && warp < 6) {
        // ---------------- epilogue: warp q owns this CTA's accumulator rows 32q .. 32q+31
        const int q = warp & 3;
        const uint32_t stg0 = sbase + P::STG_OFF + q * 2 * STG_BYTES;
        uint8_t* stg0p = smem + P::STG_OFF + q * 2 * STG_BYTES;
        int bi = 0;
        int t = 0;
        const bool residual = args.epi == DLO_EPI_RESIDUAL;
        for (int tile = pair; tile < args.num_tiles; tile += npairs, ++t) {
            const int acc = t & 1;
            const uint32_t aph = (t >> 1) & 1;
            int mb, nb;
            tile_coords(tile, args, mb, nb);
            // W8A8: the activation scale times the weight scale (epi_load)
            const float sa = (args.scales && args.act_scale) ? *args.act_scale : 1.0f;
            bool ok = mbar_wait(bar_tfull + acc * 8, aph, abort_flag);
            ok = __all_sync(0xFFFFFFFFu, ok);
            if (!ok) {
                if (lane == 0) fail();
                break;
            }
            tc_fence_after();
            const int row0 = mb * P::BM2 + static_cast<int>(rank) * BM + q * 32;
            const int row = row0 + lane;
            const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * BN;
            if (residual) {
                const float* grow = args.gate ? args.gate + static_cast<size_t>(min(row, args.M - 1) /
                                                                                 args.rows_per_batch) *
                                                                args.gate_ld
                                              : nullptr;
#pragma unroll 1
                for (int c0 = 0; c0 < BN; c0 += 32) {
                    const int col0 = nb * BN + c0;
                    if (col0 >= args.N) break;
                    EpiBS e;
                    epi_load(args, sa, col0, e);
                    float4 gv[8];
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        gv[j] = (grow && col0 + 4 * j < args.N)
                                    ? *reinterpret_cast<const float4*>(grow + col0 + 4 * j)
                                    : make_float4(1.f, 1.f, 1.f, 1.f);
                    uint32_t r[32];
                    tmem_ld_32x32b_x32_nc(taddr + c0, r);
                    tmem_wait_ld_r(r);
                    float v[32];
#pragma unroll
                    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
                    epi_apply(e, v);
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        v[4 * j] *= gv[j].x;
                        v[4 * j + 1] *= gv[j].y;
                        v[4 * j + 2] *= gv[j].z;
                        v[4 * j + 3] *= gv[j].w;
                    }
                    if (lane == 0) bulk_wait_read<1>();
                    __syncwarp();
                    uint8_t* box = stg0p + bi * STG_BYTES;
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        *reinterpret_cast<float4*>(box + sw128(lane, j)) =
                            make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        tma_reduce_add_2d(&tmO, stg0 + bi * STG_BYTES, col0, row0);
                        bulk_commit();
                    }
                    bi ^= 1;
                }
            } else {
#pragma unroll 1
                for (int c0 = 0; c0 < BN; c0 += 64) {
                    const int col0 = nb * BN + c0;
                    if (col0 >= args.N) break;
                    if (lane == 0) bulk_wait_read<1>();
                    __syncwarp();
                    uint8_t* box = stg0p + bi * STG_BYTES;
                    EpiBS e2[2];
                    epi_load(args, sa, col0, e2[0]);
                    epi_load(args, sa, col0 + 32, e2[1]);
#pragma unroll
                    for (int half = 0; half < 2; ++half) {
                        uint32_t r[32];
                        tmem_ld_32x32b_x32_nc(taddr + c0 + 32 * half, r);
                        tmem_wait_ld_r(r);
                        float v[32];
#pragma unroll
                        for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
                        epi_apply(e2[half], v);
                        if (args.epi == DLO_EPI_GELU) {
#pragma unroll
                            for (int i = 0; i < 32; ++i) v[i] = gelu_tanh(v[i]);
                        }
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            uint4 w;
                            w.x = pack_bf16x2(v[8 * j + 0], v[8 * j + 1]);
                            w.y = pack_bf16x2(v[8 * j + 2], v[8 * j + 3]);
                            w.z = pack_bf16x2(v[8 * j + 4], v[8 * j + 5]);
                            w.w = pack_bf16x2(v[8 * j + 6], v[8 * j + 7]);
                            *reinterpret_cast<uint4*>(box + sw128(lane, 4 * half + j)) = w;
                        }
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        tma_store_2d(&tmO, stg0 + bi * STG_BYTES, col0, row0);
                        bulk_commit();
                    }
                    bi ^= 1;
                }
            }
            // this CTA's accumulator rows are read: rank 0 may issue into the set again
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(tempty_r0 + acc * 8);
        }
        if (lane == 0) bulk_wait_all();
        __syncwarp();
    } else if constexpr (FP8) {
        if (warp >= 6) {
            // ---------------- e4m3 -> bf16 converters: this CTA's weight rows
            const int ct = threadIdx.x - 6 * 32;
            constexpr int kChunks = P::HALF * 8;                  // 8 codes each
            constexpr int kIter = (kChunks + kConvWarps * 32 - 1) / (kConvWarps * 32);
            int s = 0, cb = 0;
            uint32_t ph = 0, cph = 0;
            bool ok = true;
            for (int tile = pair; ok && tile < args.num_tiles; tile += npairs) {
                for (int kb = 0; kb < kblocks; ++kb) {
                    // the stage's A tile and codes have landed: the readiness
                    // signal below covers this CTA's A tile as well
                    bool got = mbar_wait(bar_full + s * 8, ph, abort_flag);
                    if (got) got = mbar_wait(bar_cempty + cb * 8, cph ^ 1, abort_flag);
                    got = __all_sync(0xFFFFFFFFu, got);
                    if (!got) {
                        if (lane == 0) fail();
                        ok = false;
                        break;
                    }
                    const uint8_t* raw = smem + P::RAW_OFF + s * P::RAW_TILE;
                    uint8_t* dst = smem + P::W_OFF + cb * P::W_TILE;
                    // every load of this thread's share first (the compiler cannot
                    // move loads above stores to a buffer it cannot tell apart)
                    uint2 v[kIter];
#pragma unroll
                    for (int j = 0; j < kIter; ++j) {
                        const int i = ct + j * kConvWarps * 32;
                        if (i < kChunks) v[j] = *reinterpret_cast<const uint2*>(raw + (i >> 3) * 64 + (i & 7) * 8);
                    }
#pragma unroll
                    for (int j = 0; j < kIter; ++j) {
                        const int i = ct + j * kConvWarps * 32;
                        if (i < kChunks) {
                            uint32_t o[4];
                            e4m3x8_to_bf16x8(v[j].x, v[j].y, o);
                            *reinterpret_cast<uint4*>(dst + sw128(i >> 3, i & 7)) =
                                make_uint4(o[0], o[1], o[2], o[3]);
                        }
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        if (rank != 0)
                            mbar_arrive(bar_wdone + cb * 8);
                        else if (ct == 0)
                            mbar_arrive_expect_tx(bar_conv + cb * 8, P::SIG_BYTES);   // rank 1's forwarded bytes
                        else
                            mbar_arrive(bar_conv + cb * 8);
                    }
                    if (++s == STAGES) {
                        s = 0;
                        ph ^= 1;
                    }
                    if (++cb == CB) {
                        cb = 0;
                        cph ^= 1;
                    }
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    // neither CTA leaves while the other may still arrive on its barriers or
    // the pair's MMAs may still read its shared memory
    cluster_sync_all();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc_pair(tmem_base, P::TMEM_COLS);
    }
}

// ------------------------------------------------------------------ host side

EncodeTiledFn get_encode() { return tensor_map_encoder(); }

// Row-major [rows, cols] matrix with row pitch ld elements of es_bytes; box of
// box_rows x box_cols, zero fill out of bounds on loads, clipping on stores.
bool make_map(CUtensorMap* m, const void* base, CUtensorMapDataType dt, int es_bytes,
              long long rows, long long cols, long long ld, int box_rows, int box_cols,
              CUtensorMapSwizzle sw) {
    EncodeTiledFn enc = get_encode();
    if (!enc) return false;
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld) * es_bytes};
    cuuint32_t box[2] = {static_cast<cuuint32_t>(box_cols), static_cast<cuuint32_t>(box_rows)};
    cuuint32_t es[2] = {1, 1};
    return enc(m, dt, 2, const_cast<void*>(base), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int g_num_sms = 0;

// Sweep order and group size of a GEMM's tiles: a group's panel of the
// re-read operand (group x the bytes of one row block of A, or of one column
// block of W) is kept within kSweepL2 bytes so it stays in L2 while the
// other operand streams past it once; the order that reads fewer DRAM bytes
// in total (the streamed operand once per group) wins.
constexpr double kSweepL2 = 40.0 * 1024 * 1024;   // of the 129 MB L2, leaving room for the streamed operand and outputs

void sweep_plan(double a_bytes, double w_bytes, int num_m, int num_n, EpiArgs* a) {
    const double a_blk = a_bytes / num_m, w_blk = w_bytes / num_n;
    int gm = static_cast<int>(kSweepL2 / (a_blk > 1.0 ? a_blk : 1.0));
    int gn = static_cast<int>(kSweepL2 / (w_blk > 1.0 ? w_blk : 1.0));
    gm = gm < 1 ? 1 : (gm > num_m ? num_m : gm);
    gn = gn < 1 ? 1 : (gn > num_n ? num_n : gn);
    const double m_sweep = a_bytes + w_bytes * ((num_m + gm - 1) / gm);
    const double n_sweep = w_bytes + a_bytes * ((num_n + gn - 1) / gn);
    a->n_major = n_sweep < m_sweep ? 1 : 0;
    a->group = a->n_major ? gn : gm;
}

template <int BN, int STAGES, bool FP8, int MT = 1, bool A8 = false, int CB = 0, int KB = 1>
cudaError_t run_gemm(const GemmParams& p, cudaStream_t s, unsigned long long* launches) {
    using PL = SmemPlan<BN, STAGES, FP8, MT, CB, KB>;
    static_assert(PL::BYTES <= 227 * 1024, "shared memory plan exceeds 227 KB");
    static bool attr_set = false;
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(gemm_kernel<BN, STAGES, FP8, MT, A8, CB, KB>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, PL::BYTES);
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    CUtensorMap ta, tb, to;
    if (A8) {
        // E4M3 codes of both operands, 128 K per box (128-byte rows)
        if (!make_map(&ta, p.A, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, p.M, p.K, p.K, BM, 128,
                      CU_TENSOR_MAP_SWIZZLE_128B) ||
            !make_map(&tb, p.W, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, p.N, p.K, p.K, BN, 128,
                      CU_TENSOR_MAP_SWIZZLE_128B))
            return cudaErrorInvalidValue;
    } else if (!make_map(&ta, p.A, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, p.M, p.K, p.K, BM, BK,
                         CU_TENSOR_MAP_SWIZZLE_128B)) {
        return cudaErrorInvalidValue;
    }
    if (A8) {
    } else if (FP8) {
        if (!make_map(&tb, p.W, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, p.N, p.K, p.K, BN, BK,
                      CU_TENSOR_MAP_SWIZZLE_NONE))
            return cudaErrorInvalidValue;
    } else if (!make_map(&tb, p.W, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, p.N, p.K, p.K, BN, BK,
                         CU_TENSOR_MAP_SWIZZLE_128B)) {
        return cudaErrorInvalidValue;
    }
    const bool residual = p.epi == DLO_EPI_RESIDUAL;
    if (!make_map(&to, p.out, residual ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                  residual ? 4 : 2, p.M, p.N, p.ldo, 32, residual ? 32 : 64, CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    EpiArgs a = {};
    a.M = p.M;
    a.N = p.N;
    a.K = p.K;
    a.epi = p.epi;
    a.bias = static_cast<const __nv_bfloat16*>(p.bias);
    a.scales = p.scales;
    a.scale_seg = p.scale_seg > 0 ? p.scale_seg : p.N;
    a.act_scale = A8 ? p.a_scale : nullptr;
    a.gate = p.gate;
    a.gate_ld = p.gate_ld;
    a.rows_per_batch = p.rows_per_batch > 0 ? p.rows_per_batch : 1;
    a.w_ready = p.w_ready ? 1 : 0;
    a.err = p.err;
    a.num_m = (p.M + MT * BM - 1) / (MT * BM);
    a.num_n = (p.N + BN - 1) / BN;
    a.num_tiles = a.num_m * a.num_n;
    sweep_plan(static_cast<double>(p.M) * p.K * (A8 ? 1 : 2), static_cast<double>(p.N) * p.K * (FP8 || A8 ? 1 : 2),
               a.num_m, a.num_n, &a);
    const int grid = a.num_tiles < g_num_sms ? a.num_tiles : g_num_sms;
    cudaError_t le_ = launch_k(gemm_kernel<BN, STAGES, FP8, MT, A8, CB, KB>, grid, PL::THREADS, PL::BYTES, s, ta, tb, to, a);
    ++*launches;
    return le_ != cudaSuccess ? le_ : cudaGetLastError();
}

// Clusters of two CTAs of gemm_pair_kernel that fit on the GPU at once
// (queried once; an SM a pair cannot use stays idle).
template <int BN, int STAGES, int CB, bool FP8, bool A8>
int pair_clusters() {
    static int n = -1;
    if (n < 0) {
        using PL = PairPlan<BN, STAGES, CB, FP8, A8>;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(2 * (g_num_sms / 2), 1, 1);
        cfg.blockDim = dim3(PL::THREADS, 1, 1);
        cfg.dynamicSmemBytes = PL::BYTES;
        cudaLaunchAttribute at[1];
        at[0].id = cudaLaunchAttributeClusterDimension;
        at[0].val.clusterDim.x = 2;
        at[0].val.clusterDim.y = 1;
        at[0].val.clusterDim.z = 1;
        cfg.attrs = at;
        cfg.numAttrs = 1;
        int c = 0;
        if (cudaOccupancyMaxActiveClusters(&c, gemm_pair_kernel<BN, STAGES, CB, FP8, A8>, &cfg) != cudaSuccess ||
            c < 1) {
            cudaGetLastError();
            c = g_num_sms / 2;
        }
        n = c;
    }
    return n;
}

template <int BN, int STAGES, int CB, bool FP8, bool A8 = false, bool WIDEN = false>
cudaError_t run_gemm_pair(const GemmParams& p, cudaStream_t s, unsigned long long* launches) {
    using PL = PairPlan<BN, STAGES, CB, FP8, A8>;
    static_assert(PL::BYTES <= 227 * 1024, "shared memory plan exceeds 227 KB");
    static bool attr_set = false;
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(gemm_pair_kernel<BN, STAGES, CB, FP8, A8, WIDEN>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, PL::BYTES);
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    CUtensorMap ta, tb, to;
    if (A8) {
        // E4M3 codes of both operands, 128 K per box (128-byte rows)
        if (!make_map(&ta, p.A, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, p.M, p.K, p.K, BM, 128,
                      CU_TENSOR_MAP_SWIZZLE_128B) ||
            !make_map(&tb, p.W, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, p.N, p.K, p.K, PL::HALF, 128,
                      CU_TENSOR_MAP_SWIZZLE_128B))
            return cudaErrorInvalidValue;
    } else {
        if (!make_map(&ta, p.A, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, p.M, p.K, p.K, BM, BK,
                      CU_TENSOR_MAP_SWIZZLE_128B))
            return cudaErrorInvalidValue;
        if (FP8 ? !make_map(&tb, p.W, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, p.N, p.K, p.K, PL::HALF, BK,
                            CU_TENSOR_MAP_SWIZZLE_NONE)
                : !make_map(&tb, p.W, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, p.N, p.K, p.K, PL::HALF, BK,
                            CU_TENSOR_MAP_SWIZZLE_128B))
            return cudaErrorInvalidValue;
    }
    const bool residual = p.epi == DLO_EPI_RESIDUAL;
    if (!make_map(&to, p.out, residual ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                  residual ? 4 : 2, p.M, p.N, p.ldo, 32, residual ? 32 : 64, CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    EpiArgs a = {};
    a.M = p.M;
    a.N = p.N;
    a.K = p.K;
    a.epi = p.epi;
    a.bias = static_cast<const __nv_bfloat16*>(p.bias);
    a.scales = p.scales;
    a.scale_seg = p.scale_seg > 0 ? p.scale_seg : p.N;
    a.act_scale = A8 ? p.a_scale : nullptr;
    a.gate = p.gate;
    a.gate_ld = p.gate_ld;
    a.rows_per_batch = p.rows_per_batch > 0 ? p.rows_per_batch : 1;
    a.w_ready = p.w_ready ? 1 : 0;
    a.err = p.err;
    a.num_m = (p.M + PL::BM2 - 1) / PL::BM2;
    a.num_n = (p.N + BN - 1) / BN;
    a.num_tiles = a.num_m * a.num_n;
    sweep_plan(static_cast<double>(p.M) * p.K * (A8 ? 1 : 2), static_cast<double>(p.N) * p.K * (FP8 || A8 ? 1 : 2),
               a.num_m, a.num_n, &a);
    const int maxc = pair_clusters<BN, STAGES, CB, FP8, A8>();
    const int pairs = a.num_tiles < maxc ? a.num_tiles : maxc;
    if (WIDEN) {
        // the codes, their widened copy (p.W) and the barrier counter
        a.wcodes = static_cast<const uint4*>(p.w_codes);
        a.wwide = static_cast<uint4*>(const_cast<void*>(p.W));
        a.wn16 = static_cast<size_t>(p.N) * p.K / 16;
        a.gbar = p.w_sync;
        cudaError_t e = cudaMemsetAsync(p.w_sync, 0, sizeof(unsigned), s);
        if (e != cudaSuccess) return e;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * pairs, 1, 1);
    cfg.blockDim = dim3(PL::THREADS, 1, 1);
    cfg.dynamicSmemBytes = PL::BYTES;
    cfg.stream = s;
    cudaLaunchAttribute at[3];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = 2;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    at[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[1].val.programmaticStreamSerializationAllowed = pdl_enabled() ? 1 : 0;
    at[2].id = cudaLaunchAttributeCooperative;   // WIDEN: the grid barrier needs every CTA resident
    at[2].val.cooperative = 1;
    cfg.attrs = at;
    cfg.numAttrs = WIDEN ? 3 : 2;
    cudaError_t le_ = cudaLaunchKernelEx(&cfg, gemm_pair_kernel<BN, STAGES, CB, FP8, A8, WIDEN>, ta, tb, to, a);
    ++*launches;
    return le_ != cudaSuccess ? le_ : cudaGetLastError();
}

// DLO_GEMM_PAIR=0 keeps every GEMM on single CTAs; =1 puts every GEMM with
// at least 256 rows on CTA pairs; unset, E4M3-weight GEMMs with 256 rows or
// more run on pairs and bf16 GEMMs follow the tile model (tuning).
int pair_mode() {
    static int v = -2;
    if (v == -2) {
        const char* e = std::getenv("DLO_GEMM_PAIR");
        v = (e && e[0] == '0' && e[1] == 0) ? 0 : (e && e[0] == '1' && e[1] == 0) ? 1 : -1;
    }
    return v;
}

// DLO_GEMM_K128=0: 128-wide bf16 tiles on 64-K stages (tuning).
bool k128_enabled() {
    static int v = -1;
    if (v < 0) {
        const char* e = std::getenv("DLO_GEMM_K128");
        v = (e && e[0] == '0' && e[1] == 0) ? 0 : 1;
    }
    return v != 0;
}

int forced_mt() {
    static int v = -1;
    if (v < 0) {
        const char* e = std::getenv("DLO_GEMM_MT");
        v = e ? std::atoi(e) : 0;
    }
    return v;
}

int forced_bn() {
    static int v = -1;
    if (v < 0) {
        const char* e = std::getenv("DLO_GEMM_BN");
        v = e ? std::atoi(e) : 0;
    }
    return v;
}

}  // namespace

namespace {

// A tensor map is a pure function of its encoding arguments, and the same
// few dozen maps (workspace, slots, resident blocks) recur every forward, so
// encoded maps are kept in a table keyed by every argument.  Encoding costs
// microseconds of host time per map; a lookup costs tens of nanoseconds.
EncodeTiledFn g_encode_raw = nullptr;

struct MapKey {
    uint64_t w[23];
    bool operator==(const MapKey& o) const { return std::memcmp(w, o.w, sizeof(w)) == 0; }
};
struct MapKeyHash {
    size_t operator()(const MapKey& k) const {
        uint64_t h = 1469598103934665603ull;   // FNV-1a over the words
        for (uint64_t v : k.w) {
            h ^= v;
            h *= 1099511628211ull;
        }
        return static_cast<size_t>(h);
    }
};
constexpr size_t kMapCacheMax = 4096;

CUresult encode_cached(CUtensorMap* m, CUtensorMapDataType dt, cuuint32_t rank, void* base,
                       const cuuint64_t* dims, const cuuint64_t* strides, const cuuint32_t* box,
                       const cuuint32_t* es, CUtensorMapInterleave il, CUtensorMapSwizzle sw,
                       CUtensorMapL2promotion l2, CUtensorMapFloatOOBfill oob) {
    if (rank < 1 || rank > 5)
        return g_encode_raw(m, dt, rank, base, dims, strides, box, es, il, sw, l2, oob);
    MapKey key;
    std::memset(key.w, 0, sizeof(key.w));
    key.w[0] = static_cast<uint64_t>(dt);
    key.w[1] = rank;
    key.w[2] = reinterpret_cast<uintptr_t>(base);
    for (cuuint32_t i = 0; i < rank; ++i) {
        key.w[3 + i] = dims[i];
        key.w[12 + i] = box[i];
        key.w[17 + i] = es[i];
    }
    for (cuuint32_t i = 0; i + 1 < rank; ++i) key.w[8 + i] = strides[i];
    key.w[22] = static_cast<uint64_t>(il) | static_cast<uint64_t>(sw) << 8 |
                static_cast<uint64_t>(l2) << 16 | static_cast<uint64_t>(oob) << 24;
    static std::mutex mu;
    static std::unordered_map<MapKey, CUtensorMap, MapKeyHash> table;
    {
        std::lock_guard<std::mutex> g(mu);
        auto it = table.find(key);
        if (it != table.end()) {
            *m = it->second;
            return CUDA_SUCCESS;
        }
    }
    const CUresult r = g_encode_raw(m, dt, rank, base, dims, strides, box, es, il, sw, l2, oob);
    if (r == CUDA_SUCCESS) {
        std::lock_guard<std::mutex> g(mu);
        if (table.size() >= kMapCacheMax) table.clear();
        table.emplace(key, *m);
    }
    return r;
}

}  // namespace

EncodeTiledFn tensor_map_encoder() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess) {
            g_encode_raw = reinterpret_cast<EncodeTiledFn>(p);
            fn = encode_cached;
        }
    });
    return fn;
}

int gemm_num_sms() {
    if (!g_num_sms) {
        int dev = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&g_num_sms, cudaDevAttrMultiProcessorCount, dev);
        if (g_num_sms <= 0) g_num_sms = 1;
    }
    return g_num_sms;
}

cudaError_t launch_widen_e4m3(const void* codes, size_t n, void* out, cudaStream_t s,
                              unsigned long long* launches) {
    if (n == 0) return cudaSuccess;
    if ((reinterpret_cast<uintptr_t>(codes) | reinterpret_cast<uintptr_t>(out)) & 15) return cudaErrorInvalidValue;
    const size_t n16 = n / 16;
    const int tail = static_cast<int>(n % 16);
    const cudaError_t e = launch_k(widen_e4m3_kernel, gemm_num_sms() * 4, 256, 0, s,
                                   static_cast<const uint4*>(codes), static_cast<uint4*>(out), n16,
                                   static_cast<const uint8_t*>(codes) + n16 * 16,
                                   static_cast<uint16_t*>(out) + n16 * 16, tail);
    ++*launches;
    return e != cudaSuccess ? e : cudaGetLastError();
}

namespace {

// bf16 and W8A8 GEMMs: single CTAs (128-row tiles) or CTA pairs (256-row
// tiles), and the N tile, from the cost of one 128-byte-wide K step per SM
// times the waves of tiles.  Single CTAs: SM cycles measured on GB300 while
// every SM streams its operands from L2 (a step moves 16 KB of A and BN x 128
// bytes of weights into the SM, which takes in ~70 bytes per cycle).  Pairs:
// an SM takes in only BN/2 weight rows, but its MMAs also read the peer's
// half; their costs are set from graph-timed runs of both kernels at 2048-
// and 8192-row shapes (pairs 11-15% faster at 8192 rows, 0-4% slower at
// 2048), so pairs win where many waves of wide tiles run.  128-wide bf16
// single-CTA tiles on 128-K stages take 433 cycles per 64 K (measured the
// same way).  A W8A8 step (128
// K of E4M3, MMAs at twice the bf16 rate) has the bf16 step's bytes and
// cycles.  DLO_GEMM_BN forces the width, DLO_GEMM_PAIR=0 or 1 single CTAs or
// pairs (tuning).
void pick_tile(const GemmParams& p, int* bn, bool* pair) {
    const int widths[3] = {128, 192, 256};
    const bool k128 = p.a_dtype == DLO_DT_BF16 && k128_enabled();
    const double single_cyc[3] = {k128 ? 433.0 : 509.0, 543, 651};
    const double pair_cyc[3] = {530, 580, 600};
    const long long num_m = (p.M + BM - 1) / BM;
    const int max_pairs = g_num_sms / 2 > 0 ? g_num_sms / 2 : 1;
    const bool pairs_ok = pair_mode() != 0 && p.M >= 2 * BM;
    const bool singles_ok = !(pair_mode() == 1 && pairs_ok);
    double best = 0;
    *bn = 256;
    *pair = false;
    for (int i = 0; i < 3; ++i) {
        const int w = widths[i];
        if (forced_bn() > 0 && forced_bn() != w) continue;
        const long long nn = (p.N + w - 1) / w;
        const double t1 = static_cast<double>((num_m * nn + g_num_sms - 1) / g_num_sms) * single_cyc[i];
        if (singles_ok && (best == 0 || t1 < best)) {
            best = t1;
            *bn = w;
            *pair = false;
        }
        if (pairs_ok) {
            const long long tiles = ((p.M + 2 * BM - 1) / (2 * BM)) * nn;
            const double t2 = static_cast<double>((tiles + max_pairs - 1) / max_pairs) * pair_cyc[i];
            if (best == 0 || t2 < best) {
                best = t2;
                *bn = w;
                *pair = true;
            }
        }
    }
}

}  // namespace

namespace {

// W8A16 with the widening inside the bf16 pair GEMM (GemmParams::w_codes).
// cudaErrorNotSupported when this GEMM or this driver cannot take that form;
// the caller then widens with launch_widen_e4m3 and runs launch_gemm.  The
// cooperative cluster launch is first tried outside a stream capture; if the
// driver refuses it, the form is not tried again in this process.
std::atomic<int> g_widen_in_gemm{-1};   // -1 not tried, 0 refused (or DLO_WIDEN_IN_GEMM=0), 1 works

cudaError_t launch_gemm_widen(const GemmParams& p, cudaStream_t s, unsigned long long* launches) {
    if (g_widen_in_gemm < 0) {
        // DLO_WIDEN_IN_GEMM=0: always the separate widening kernel (tuning;
        // also the form a profiler can replay)
        const char* e = std::getenv("DLO_WIDEN_IN_GEMM");
        if (e && e[0] == '0' && e[1] == 0) g_widen_in_gemm = 0;
    }
    if (g_widen_in_gemm == 0 || !p.w_sync || p.w_dtype != DLO_DT_BF16 || p.a_dtype != DLO_DT_BF16)
        return cudaErrorNotSupported;
    const size_t nk = static_cast<size_t>(p.N) * p.K;
    if (nk % 16 || ((reinterpret_cast<uintptr_t>(p.w_codes) | reinterpret_cast<uintptr_t>(p.W)) & 15))
        return cudaErrorNotSupported;
    int bn = 256;
    bool pair = false;
    pick_tile(p, &bn, &pair);
    if (!pair || bn != 256) return cudaErrorNotSupported;
    if (g_widen_in_gemm < 0) {
        cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
        if (cudaStreamIsCapturing(s, &cs) != cudaSuccess || cs != cudaStreamCaptureStatusNone)
            return cudaErrorNotSupported;
    }
    const cudaError_t e = run_gemm_pair<256, 6, 0, false, false, true>(p, s, launches);
    if (e != cudaSuccess) {
        cudaGetLastError();
        if (g_widen_in_gemm < 0) {
            g_widen_in_gemm = 0;
            return cudaErrorNotSupported;
        }
        return e;
    }
    g_widen_in_gemm = 1;
    return cudaSuccess;
}

}  // namespace

cudaError_t launch_gemm(const GemmParams& p, cudaStream_t s, unsigned long long* launches) {
    if (p.M <= 0) return cudaSuccess;
    gemm_num_sms();
    if (p.w_codes) return launch_gemm_widen(p, s, launches);
    // Single-CTA E4M3-weight GEMMs: N tile from a small cost model, time ~
    // waves x tile width / efficiency, where narrower tiles move more
    // shared-memory bytes per FLOP (128-wide tiles are limited to about 3/4
    // of the MMA rate, 192-wide to ~0.95).  DLO_GEMM_BN=128|192|256 forces
    // one (tuning).
    const long long num_m = (p.M + BM - 1) / BM;
    auto cost = [&](int bn) {
        const long long tiles = num_m * ((p.N + bn - 1) / bn);
        const double eff = bn == 256 ? 1.0 : bn == 192 ? 0.95 : 0.75;
        return static_cast<double>((tiles + g_num_sms - 1) / g_num_sms) * bn / eff;
    };
    int bn = 256;
    if (cost(192) < cost(bn)) bn = 192;
    if (cost(128) < cost(bn)) bn = 128;
    if (forced_bn() == 128 || forced_bn() == 192 || forced_bn() == 256) bn = forced_bn();
    if (p.w_dtype == DLO_DT_E4M3 && p.a_dtype != DLO_DT_E4M3) {
        // E4M3 with at least one full 256-row pair tile: CTA pairs, 256 x 256
        // tiles, one M = 256 MMA over both SMs (gemm_pair_kernel)
        if (pair_mode() != 0 && p.M >= 2 * BM) return run_gemm_pair<256, 6, 3, true>(p, s, launches);
        // E4M3: 256-row CTA tiles (two 128-row accumulators) share each
        // widened weight tile, halving the widening work per FLOP, when
        // there are enough row blocks to fill the SMs.  DLO_GEMM_MT=1 turns
        // it off (tuning).
        const long long tiles2 = ((p.M + 255) / 256) * ((p.N + 127) / 128);
        if (forced_mt() != 1 && (forced_mt() == 2 || tiles2 >= g_num_sms))
            return run_gemm<128, 4, true, 2, false, 2>(p, s, launches);
        if (bn == 256) return run_gemm<256, 3, true>(p, s, launches);
        if (bn == 192) return run_gemm<192, 3, true>(p, s, launches);
        return run_gemm<128, 4, true>(p, s, launches);
    }
    if (p.a_dtype == DLO_DT_E4M3) {
        // W8A8: both operands E4M3; same stage bytes as bf16
        if (p.w_dtype != DLO_DT_E4M3 || !p.a_scale || !p.scales) return cudaErrorInvalidValue;
        int w8_bn = 256;
        bool w8_pair = false;
        pick_tile(p, &w8_bn, &w8_pair);
        if (w8_pair) {
            if (w8_bn == 256) return run_gemm_pair<256, 6, 0, false, true>(p, s, launches);
            if (w8_bn == 192) return run_gemm_pair<192, 6, 0, false, true>(p, s, launches);
            return run_gemm_pair<128, 7, 0, false, true>(p, s, launches);
        }
        if (w8_bn == 256) return run_gemm<256, 4, false, 1, true>(p, s, launches);
        if (w8_bn == 192) return run_gemm<192, 4, false, 1, true>(p, s, launches);
        return run_gemm<128, 6, false, 1, true>(p, s, launches);
    }
    if (p.w_dtype != DLO_DT_BF16) return cudaErrorNotSupported;
    int best_bn = 256;
    bool best_pair = false;
    pick_tile(p, &best_bn, &best_pair);
    if (best_pair) {
        if (best_bn == 256) return run_gemm_pair<256, 6, 0, false>(p, s, launches);
        if (best_bn == 192) return run_gemm_pair<192, 6, 0, false>(p, s, launches);
        return run_gemm_pair<128, 7, 0, false>(p, s, launches);
    }
    if (best_bn == 256) return run_gemm<256, 4, false>(p, s, launches);
    if (best_bn == 192) return run_gemm<192, 4, false>(p, s, launches);
    // 128-wide tiles: 128-K stages (two boxes per operand, three stages)
    // halve the stage hand-overs per K; DLO_GEMM_K128=0 keeps 64-K stages
    if (k128_enabled()) return run_gemm<128, 3, false, 1, false, 0, 2>(p, s, launches);
    return run_gemm<128, 6, false>(p, s, launches);
}

}  // namespace dlo

// ====================================================================== no-allocation GEMM
//
// dlo_op_gemm writes its device error word into memory the caller allocated.
// Callers that cannot allocate device memory at all use dlo_op_gemm_noalloc
// instead: its scratch -- the same error word -- lives in the static device
// array below, which every GPU that loads this library holds until the
// process exits.

namespace {

constexpr size_t kNoAllocScratchBytes = 256;   // stated maximum scratch size
constexpr size_t kNoAllocNeedBytes = sizeof(int);
constexpr int kNoAllocMaxDevices = 64;
static_assert(kNoAllocNeedBytes <= kNoAllocScratchBytes, "the GEMM's scratch must fit the static array");

}  // namespace

static __device__ __align__(256) int g_noalloc_scratch[kNoAllocScratchBytes / sizeof(int)];

namespace {

std::mutex g_noalloc_mu;
int* g_noalloc_ptr[kNoAllocMaxDevices] = {};

// Device address of the static scratch on the current device, looked up once
// per device (the host-side name is only a stand-in, never a device address).
cudaError_t noalloc_scratch(int** ptr_out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kNoAllocMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    if (!g_noalloc_ptr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return e;
        g_noalloc_ptr[dev] = static_cast<int*>(p);
    }
    *ptr_out = g_noalloc_ptr[dev];
    return cudaSuccess;
}

}  // namespace

extern "C" dlo_status dlo_op_gemm_noalloc(const void* A, const void* W, int w_dtype,
                                          const float* scales, int scale_seg, const void* bias,
                                          int M, int N, int K, int epilogue, void* out, int ldo,
                                          const float* gate, int gate_ld, int rows_per_batch,
                                          void* stream) {
    // the same checks and parameters as dlo_op_gemm; only the error word differs
    dlo::GemmParams p;
    dlo_status r = dlo::op_gemm_params(A, W, w_dtype, scales, scale_seg, bias, M, N, K, epilogue, out, ldo,
                                       gate, gate_ld, rows_per_batch, DLO_DT_BF16, nullptr, &p);
    if (r != DLO_OK) return r;
    int* scratch = nullptr;
    cudaError_t e = noalloc_scratch(&scratch);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return dlo::op_fail(DLO_ECUDA, std::string("static scratch lookup: ") + cudaGetErrorString(e));
    }
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // the array keeps the previous call's contents: the error word starts at 0
    e = cudaMemsetAsync(scratch, 0, kNoAllocNeedBytes, s);
    if (e != cudaSuccess) return dlo::op_result(e);
    p.err = scratch;
    return dlo::op_launch_gemm(p, s);
}
