// Bandwidth-bound kernels of one block: LayerNorm (+adaLN modulate or affine),
// RMSNorm on q/k, the adaLN GEMV SiLU(c) W^T + b, the video modulation add,
// dtype conversions of the carried hidden state, and the zero-copy slot
// gather that reads mapped host memory with 16-byte loads.
//
// One warp per row for the row-wise kernels.
#include <cuda_bf16.h>

#include <cstdlib>

#include "internal.h"
#include "ptx.cuh"

namespace dlo {

bool pdl_enabled() {
    static int v = -1;
    if (v < 0) {
        const char* e = std::getenv("DLO_PDL");
        v = (e && e[0] == '0') ? 0 : 1;
    }
    return v != 0;
}

namespace {

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
    return v;
}

__device__ __forceinline__ float bf(const __nv_bfloat16 v) { return __bfloat162float(v); }

// out = LN(x) * (1 + scale) + shift | LN(x) * w + b | LN(x)
// WPR warps per row (a row group); each thread holds V4 float4 of the row in
// registers, mean and variance come from the registers (two passes, warp
// shuffles then shared memory across the row group), so HBM sees one read of
// x and one write of the bf16 output.  The launcher uses two warps per row,
// more only for rows too wide for 20 float4 per thread.
template <int V4, int WPR>
__global__ void __launch_bounds__(256) layernorm_kernel(const float* __restrict__ x, int rows,
                                                        int D, int rpb,
                                                        const float* __restrict__ shift,
                                                        const float* __restrict__ scale,
                                                        int mod_ld,
                                                        const __nv_bfloat16* __restrict__ w,
                                                        const __nv_bfloat16* __restrict__ b,
                                                        float eps,
                                                        __nv_bfloat16* __restrict__ out) {
    pdl_wait();
    pdl_launch_dependents();
    constexpr int RPC = 8 / WPR;                  // rows per 256-thread CTA
    constexpr bool kPre = V4 <= 16;               // modulation prefetched into registers
    __shared__ float red[2][8];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int sub = warp % WPR;
    const int row = blockIdx.x * RPC + warp / WPR;
    const bool live = row < rows;
    const int n4 = D >> 2;
    const int t0 = sub * 32 + lane;               // first float4 of this thread
    const float4* xr = reinterpret_cast<const float4*>(x + static_cast<size_t>(live ? row : 0) * D);
    float4 v[V4];
#pragma unroll
    for (int j = 0; j < V4; ++j) {
        const int i = t0 + 32 * WPR * j;
        v[j] = (live && i < n4) ? xr[i] : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    const int bt = (live ? row : 0) / rpb;
    float4 sc4[kPre ? V4 : 1], sh4[kPre ? V4 : 1];
    if constexpr (kPre) {
#pragma unroll
        for (int j = 0; j < V4; ++j) {
            const int i = t0 + 32 * WPR * j;
            sc4[j] = make_float4(0.f, 0.f, 0.f, 0.f);
            sh4[j] = sc4[j];
            if (live && i < n4 && scale) {
                sc4[j] = *reinterpret_cast<const float4*>(scale + static_cast<size_t>(bt) * mod_ld + i * 4);
                sh4[j] = *reinterpret_cast<const float4*>(shift + static_cast<size_t>(bt) * mod_ld + i * 4);
            }
        }
    }
    float sum = 0.f;
#pragma unroll
    for (int j = 0; j < V4; ++j) sum += (v[j].x + v[j].y) + (v[j].z + v[j].w);
    sum = warp_sum(sum);
    if constexpr (WPR > 1) {
        if (lane == 0) red[0][warp] = sum;
        __syncthreads();
        sum = 0.f;
#pragma unroll
        for (int k = 0; k < WPR; ++k) sum += red[0][warp - sub + k];
    }
    const float mean = sum / static_cast<float>(D);
    float q = 0.f;
#pragma unroll
    for (int j = 0; j < V4; ++j) {
        if (t0 + 32 * WPR * j < n4) {
            const float a = v[j].x - mean, bb = v[j].y - mean, c = v[j].z - mean, d = v[j].w - mean;
            q += (a * a + bb * bb) + (c * c + d * d);
        }
    }
    q = warp_sum(q);
    if constexpr (WPR > 1) {
        if (lane == 0) red[1][warp] = q;
        __syncthreads();
        q = 0.f;
#pragma unroll
        for (int k = 0; k < WPR; ++k) q += red[1][warp - sub + k];
    }
    if (!live) return;
    const float var = q / static_cast<float>(D);
    const float rstd = rsqrtf(var + eps);
    uint2* orow = reinterpret_cast<uint2*>(out + static_cast<size_t>(row) * D);
#pragma unroll
    for (int j = 0; j < V4; ++j) {
        const int i = t0 + 32 * WPR * j;
        if (i >= n4) continue;
        float y0 = (v[j].x - mean) * rstd, y1 = (v[j].y - mean) * rstd;
        float y2 = (v[j].z - mean) * rstd, y3 = (v[j].w - mean) * rstd;
        const int d = i * 4;
        if (scale) {
            float4 sc, sh;
            if constexpr (kPre) {
                sc = sc4[j];
                sh = sh4[j];
            } else {
                sc = *reinterpret_cast<const float4*>(scale + static_cast<size_t>(bt) * mod_ld + d);
                sh = *reinterpret_cast<const float4*>(shift + static_cast<size_t>(bt) * mod_ld + d);
            }
            y0 = y0 * (1.f + sc.x) + sh.x;
            y1 = y1 * (1.f + sc.y) + sh.y;
            y2 = y2 * (1.f + sc.z) + sh.z;
            y3 = y3 * (1.f + sc.w) + sh.w;
        } else if (w) {
            const uint2 wv = *reinterpret_cast<const uint2*>(w + d);
            const uint2 bv = *reinterpret_cast<const uint2*>(b + d);
            const float2 w01 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&wv.x));
            const float2 w23 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&wv.y));
            const float2 b01 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&bv.x));
            const float2 b23 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&bv.y));
            y0 = y0 * w01.x + b01.x;
            y1 = y1 * w01.y + b01.y;
            y2 = y2 * w23.x + b23.x;
            y3 = y3 * w23.y + b23.y;
        }
        uint2 o;
        o.x = pack_bf16x2(y0, y1);
        o.y = pack_bf16x2(y2, y3);
        orow[i] = o;
    }
}

// x[row, col0 + d] = x * rsqrt(mean(x^2) + eps) * w[d], in place, bf16; up to
// two column segments of the same rows (q and k).
__global__ void __launch_bounds__(256) rmsnorm_kernel(__nv_bfloat16* __restrict__ x, int rows,
                                                      int D, int ld, int col0a,
                                                      const __nv_bfloat16* __restrict__ wa,
                                                      int col0b,
                                                      const __nv_bfloat16* __restrict__ wb,
                                                      float eps) {
    pdl_wait();
    pdl_launch_dependents();
    const int gw = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    const int nseg = wb ? 2 : 1;
    if (gw >= rows * nseg) return;
    const int row = gw / nseg, seg = gw % nseg;
    const int col0 = seg ? col0b : col0a;
    const __nv_bfloat16* w = seg ? wb : wa;
    uint4* xr = reinterpret_cast<uint4*>(x + static_cast<size_t>(row) * ld + col0);
    const int n8 = D >> 3;
    float s = 0.f;
    for (int i = lane; i < n8; i += 32) {
        const uint4 v = xr[i];
        const __nv_bfloat162* p = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float2 f = __bfloat1622float2(p[j]);
            s += f.x * f.x + f.y * f.y;
        }
    }
    const float r = rsqrtf(warp_sum(s) / static_cast<float>(D) + eps);
    const uint4* wr = reinterpret_cast<const uint4*>(w);
    for (int i = lane; i < n8; i += 32) {
        uint4 v = xr[i];
        const uint4 g = wr[i];
        __nv_bfloat162* p = reinterpret_cast<__nv_bfloat162*>(&v);
        const __nv_bfloat162* gp = reinterpret_cast<const __nv_bfloat162*>(&g);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float2 f = __bfloat1622float2(p[j]);
            const float2 gg = __bfloat1622float2(gp[j]);
            p[j] = __floats2bfloat162_rn(f.x * r * gg.x, f.y * r * gg.y);
        }
        xr[i] = v;
    }
}

// m[b, n] = sum_i SiLU(c[b, i]) W[n, i] + bias[n].
// SiLU(c) of up to BC batch rows x ADALN_CCH columns is computed once per CTA
// into shared memory; each warp owns ROWS consecutive output rows and, per
// step, issues ROWS x ADALN_U 16-byte W loads (streaming, evict-first) before
// their FMAs, so the bytes in flight stream W (a third of a DiT block) at HBM
// rate; 5 x 256 columns per step cover a 1152-wide conditioning in one step.
// ROWS is chosen on the host so that the whole grid is resident at once (one
// wave).  W_READY: W is not written by the preceding kernel in the stream
// (block weights staged, and waited for, before the block's first kernel),
// so the first step's W loads are issued before the programmatic-launch wait
// and overlap the predecessor's tail; c and m are touched only after it.
// Those early loads read L2 (.cg): the slot held other weights two blocks
// ago and this SM's L1 may still hold lines of them.
constexpr int ADALN_CCH = 2048;   // columns of SiLU(c) held in shared memory
constexpr int ADALN_U = 5;        // 256-column steps unrolled per iteration

template <int ROWS, bool L2ONLY>
__device__ __forceinline__ void adaln_load_w(const __nv_bfloat16* __restrict__ W, int C, int N, int n0,
                                             int c0, int n8, int i0, uint4 (&wv)[ADALN_U][ROWS]) {
#pragma unroll
    for (int u = 0; u < ADALN_U; ++u) {
        const int i = i0 + 32 * u;
#pragma unroll
        for (int r = 0; r < ROWS; ++r) {
            const int n = n0 + r;
            const uint4* src = reinterpret_cast<const uint4*>(W + static_cast<size_t>(n) * C + c0) + i;
            wv[u][r] = (i < n8 && n < N) ? (L2ONLY ? __ldcg(src) : __ldcs(src)) : make_uint4(0, 0, 0, 0);
        }
    }
}

template <int BC, int ROWS, bool W_READY>
__global__ void __launch_bounds__(256) adaln_kernel(const __nv_bfloat16* __restrict__ c, int B,
                                                    int C, const __nv_bfloat16* __restrict__ W,
                                                    const __nv_bfloat16* __restrict__ bias,
                                                    int N, float* __restrict__ m) {
    if (!W_READY) {
        pdl_wait();
        pdl_launch_dependents();
    }
    extern __shared__ float sc[];   // [BC][ADALN_CCH]
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n0 = (blockIdx.x * 8 + warp) * ROWS;
    bool waited = !W_READY;
    for (int b0 = 0; b0 < B; b0 += BC) {
        const int nb = min(BC, B - b0);
        float acc[ROWS][BC];
#pragma unroll
        for (int r = 0; r < ROWS; ++r)
#pragma unroll
            for (int j = 0; j < BC; ++j) acc[r][j] = 0.f;
        for (int c0 = 0; c0 < C; c0 += ADALN_CCH) {
            const int cn = min(ADALN_CCH, C - c0);
            const int n8 = cn >> 3;   // 16-byte W chunks per row in this column chunk
            uint4 wv[ADALN_U][ROWS];
            if (!waited)
                adaln_load_w<ROWS, true>(W, C, N, n0, c0, n8, lane, wv);
            else
                adaln_load_w<ROWS, false>(W, C, N, n0, c0, n8, lane, wv);
            if (!waited) {
                pdl_wait();             // c may come from, and m is read by, neighbours
                pdl_launch_dependents();
                waited = true;
            }
            __syncthreads();
            for (int i = threadIdx.x; i < BC * cn; i += blockDim.x) {
                const int bb = i / cn, cc = i - bb * cn;
                float v = 0.f;
                if (bb < nb) {
                    v = __bfloat162float(c[static_cast<size_t>(b0 + bb) * C + c0 + cc]);
                    v = v / (1.f + __expf(-v));
                }
                sc[bb * ADALN_CCH + cc] = v;
            }
            __syncthreads();
            for (int i0 = lane; i0 < n8; i0 += 32 * ADALN_U) {
                if (i0 != lane) adaln_load_w<ROWS, false>(W, C, N, n0, c0, n8, i0, wv);
#pragma unroll
                for (int u = 0; u < ADALN_U; ++u) {
                    const int i = i0 + 32 * u;
                    if (i < n8) {
#pragma unroll
                        for (int bb = 0; bb < BC; ++bb) {
                            const float4 s0 = *reinterpret_cast<const float4*>(&sc[bb * ADALN_CCH + i * 8]);
                            const float4 s1 = *reinterpret_cast<const float4*>(&sc[bb * ADALN_CCH + i * 8 + 4]);
#pragma unroll
                            for (int r = 0; r < ROWS; ++r) {
                                const __nv_bfloat162* wp = reinterpret_cast<const __nv_bfloat162*>(&wv[u][r]);
                                const float2 w0 = __bfloat1622float2(wp[0]), w1 = __bfloat1622float2(wp[1]);
                                const float2 w2 = __bfloat1622float2(wp[2]), w3 = __bfloat1622float2(wp[3]);
                                acc[r][bb] += s0.x * w0.x + s0.y * w0.y + s0.z * w1.x + s0.w * w1.y +
                                              s1.x * w2.x + s1.y * w2.y + s1.z * w3.x + s1.w * w3.y;
                            }
                        }
                    }
                }
            }
        }
        if (!waited) {
            pdl_wait();
            pdl_launch_dependents();
            waited = true;
        }
#pragma unroll
        for (int r = 0; r < ROWS; ++r) {
#pragma unroll
            for (int bb = 0; bb < BC; ++bb) {
                const float v = warp_sum(acc[r][bb]);
                const int n = n0 + r;
                if (lane == 0 && bb < nb && n < N)
                    m[static_cast<size_t>(b0 + bb) * N + n] = v + __bfloat162float(bias[n]);
            }
        }
    }
}

// m[b, r] = e[b, r] + table[r] over r < 6D
__global__ void mod_add_kernel(const float* __restrict__ e, const __nv_bfloat16* __restrict__ t,
                               int B, int n6d, float* __restrict__ m) {
    pdl_wait();
    pdl_launch_dependents();
    const size_t i = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (i >= static_cast<size_t>(B) * n6d) return;
    m[i] = e[i] + bf(t[i % n6d]);
}

__global__ void bf16_to_f32_kernel(const __nv_bfloat16* __restrict__ in, float* __restrict__ out,
                                   size_t n8) {
    pdl_wait();
    pdl_launch_dependents();
    const size_t i = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (i >= n8) return;
    const uint4 v = reinterpret_cast<const uint4*>(in)[i];
    const __nv_bfloat162* p = reinterpret_cast<const __nv_bfloat162*>(&v);
    float4 a, b;
    float2 f0 = __bfloat1622float2(p[0]), f1 = __bfloat1622float2(p[1]);
    float2 f2 = __bfloat1622float2(p[2]), f3 = __bfloat1622float2(p[3]);
    a = make_float4(f0.x, f0.y, f1.x, f1.y);
    b = make_float4(f2.x, f2.y, f3.x, f3.y);
    reinterpret_cast<float4*>(out)[2 * i] = a;
    reinterpret_cast<float4*>(out)[2 * i + 1] = b;
}

__global__ void f32_to_bf16_kernel(const float* __restrict__ in, __nv_bfloat16* __restrict__ out,
                                   size_t n8) {
    pdl_wait();
    pdl_launch_dependents();
    const size_t i = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (i >= n8) return;
    const float4 a = reinterpret_cast<const float4*>(in)[2 * i];
    const float4 b = reinterpret_cast<const float4*>(in)[2 * i + 1];
    uint4 o;
    o.x = pack_bf16x2(a.x, a.y);
    o.y = pack_bf16x2(a.z, a.w);
    o.z = pack_bf16x2(b.x, b.y);
    o.w = pack_bf16x2(b.z, b.w);
    reinterpret_cast<uint4*>(out)[i] = o;
}

// dst[i] = src[i] over 16-byte words; src may be mapped host memory.  Four
// independent loads per thread are in flight before the stores.
// ---- dynamic per-tensor E4M3 quantisation of an activation (W8A8 linears)
//
// s = amax|x| / 448 in fp32 (1 when amax = 0), r = 1 / s rounded to fp32;
// code = E4M3_rn_satfinite(x * r) with the product rounded to fp32 (the
// inverted-scale form: one multiply per element).  Two launches: partial maxima per CTA,
// then every CTA of the quantiser reduces the partials itself (no atomics,
// no memset, deterministic) before it converts its share of the tensor.

// max over the 16-bit halves of |bf16| bit patterns: for non-negative values
// the bit order is the numeric order, and NaN patterns sort above infinity.
__device__ __forceinline__ uint32_t absmax_bf16x8(uint32_t m, const uint4& v) {
    m = __vmaxu2(m, v.x & 0x7FFF7FFFu);
    m = __vmaxu2(m, v.y & 0x7FFF7FFFu);
    m = __vmaxu2(m, v.z & 0x7FFF7FFFu);
    m = __vmaxu2(m, v.w & 0x7FFF7FFFu);
    return m;
}

__device__ __forceinline__ uint32_t block_max_u32(uint32_t m, uint32_t* sh) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
    if ((threadIdx.x & 31) == 0) sh[threadIdx.x >> 5] = m;
    __syncthreads();
    if (threadIdx.x < 32) {
        m = threadIdx.x < (blockDim.x >> 5) ? sh[threadIdx.x] : 0u;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
        if (threadIdx.x == 0) sh[0] = m;
    }
    __syncthreads();
    return sh[0];
}

// Element chunk i (8 bf16) of a [rows, 8 * c8] tensor with row stride ld:
// contiguous tensors (ld == 8 * c8) are addressed flat, without a division.
__device__ __forceinline__ const uint4* chunk_ptr(const __nv_bfloat16* x, long long i, int c8, int ld,
                                                  bool flat) {
    if (flat) return reinterpret_cast<const uint4*>(x) + i;
    const long long r = i / c8;
    return reinterpret_cast<const uint4*>(x + r * ld + (i - r * c8) * 8);
}

constexpr int kQU = 4;   // chunks in flight per thread

__global__ void __launch_bounds__(256) amax_partial_kernel(const __nv_bfloat16* __restrict__ x,
                                                           int rows, int c8, int ld,
                                                           float* __restrict__ part) {
    pdl_wait();
    pdl_launch_dependents();
    __shared__ uint32_t sh[32];
    uint32_t m = 0;
    const long long n = 1LL * rows * c8;
    const bool flat = ld == 8 * c8;
    const long long stride = gridDim.x * 256LL;
    long long i = blockIdx.x * 256LL + threadIdx.x;
    for (; i + (kQU - 1) * stride < n; i += kQU * stride) {
        uint4 v[kQU];
#pragma unroll
        for (int u = 0; u < kQU; ++u) v[u] = *chunk_ptr(x, i + u * stride, c8, ld, flat);
#pragma unroll
        for (int u = 0; u < kQU; ++u) m = absmax_bf16x8(m, v[u]);
    }
    for (; i < n; i += stride) m = absmax_bf16x8(m, *chunk_ptr(x, i, c8, ld, flat));
    m = max(m & 0xFFFFu, m >> 16);
    m = block_max_u32(m, sh);
    if (threadIdx.x == 0) part[blockIdx.x] = __uint_as_float(m << 16);
}

__device__ __forceinline__ uint2 e4m3x8(const uint4& v, float inv) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t o[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const float f0 = __uint_as_float(w[2 * h] << 16), f1 = __uint_as_float(w[2 * h] & 0xFFFF0000u);
        const float f2 = __uint_as_float(w[2 * h + 1] << 16),
                    f3 = __uint_as_float(w[2 * h + 1] & 0xFFFF0000u);
        o[h] = e4m3x2_rn_sat(__fmul_rn(f0, inv), __fmul_rn(f1, inv)) |
               (e4m3x2_rn_sat(__fmul_rn(f2, inv), __fmul_rn(f3, inv)) << 16);
    }
    return make_uint2(o[0], o[1]);
}

__global__ void __launch_bounds__(256) quant_e4m3_kernel(const __nv_bfloat16* __restrict__ x,
                                                         int rows, int c8, int ld,
                                                         const float* __restrict__ part, int nparts,
                                                         uint8_t* __restrict__ q,
                                                         float* __restrict__ scale_out) {
    pdl_wait();
    pdl_launch_dependents();
    __shared__ uint32_t sh[32];
    uint32_t m = 0;
    for (int i = threadIdx.x; i < nparts; i += 256) m = max(m, __float_as_uint(part[i]));
    m = block_max_u32(m, sh);
    const float amax = __uint_as_float(m);
    const float s = amax == 0.0f ? 1.0f : __fdiv_rn(amax, 448.0f);
    const float inv = __frcp_rn(s);
    if (blockIdx.x == 0 && threadIdx.x == 0) *scale_out = s;
    const long long n = 1LL * rows * c8;
    const bool flat = ld == 8 * c8;
    const long long stride = gridDim.x * 256LL;
    uint2* qo = reinterpret_cast<uint2*>(q);   // codes are contiguous: chunk i -> 8 bytes at 8 i
    long long i = blockIdx.x * 256LL + threadIdx.x;
    for (; i + (kQU - 1) * stride < n; i += kQU * stride) {
        uint4 v[kQU];
#pragma unroll
        for (int u = 0; u < kQU; ++u) v[u] = *chunk_ptr(x, i + u * stride, c8, ld, flat);
#pragma unroll
        for (int u = 0; u < kQU; ++u) qo[i + u * stride] = e4m3x8(v[u], inv);
    }
    for (; i < n; i += stride) qo[i] = e4m3x8(*chunk_ptr(x, i, c8, ld, flat), inv);
}

// A wait that nothing completes: one thread waits (bounded, with the limit
// every kernel of this library uses) on an mbarrier that never receives its
// arrival, then records the time-out in the error word and exits -- the path
// any kernel takes when one of its waits runs out, exercised without a fault.
__global__ void wait_selftest_kernel(int* __restrict__ err) {
    pdl_wait();
    pdl_launch_dependents();
    __shared__ __align__(8) unsigned long long bar;
    if (threadIdx.x != 0) return;
    const uint32_t b = smem_u32(&bar);
    mbar_init(b, 1);
    fence_mbar_init();
    if (!mbar_wait(b, 0, nullptr)) atomicExch(err, 1);
}

__global__ void __launch_bounds__(1024) gather_kernel(uint4* __restrict__ dst,
                                                      const uint4* __restrict__ src, size_t n16) {
    const size_t stride = static_cast<size_t>(gridDim.x) * blockDim.x;
    size_t i = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    for (; i + 3 * stride < n16; i += 4 * stride) {
        const uint4 a = src[i];
        const uint4 b = src[i + stride];
        const uint4 c = src[i + 2 * stride];
        const uint4 d = src[i + 3 * stride];
        dst[i] = a;
        dst[i + stride] = b;
        dst[i + 2 * stride] = c;
        dst[i + 3 * stride] = d;
    }
    for (; i < n16; i += stride) dst[i] = src[i];
}

// *out += sum of 64-bit words (mod 2^64): reads every byte of a staged slot,
// so it is the "compute" of an opaque bytes block.
__global__ void __launch_bounds__(256) checksum_kernel(const uint4* __restrict__ src, size_t n16,
                                                       unsigned long long* __restrict__ out) {
    pdl_wait();
    pdl_launch_dependents();
    const size_t stride = static_cast<size_t>(gridDim.x) * blockDim.x;
    unsigned long long s = 0;
    for (size_t i = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n16; i += stride) {
        const uint4 v = src[i];
        s += (static_cast<unsigned long long>(v.y) << 32) | v.x;
        s += (static_cast<unsigned long long>(v.w) << 32) | v.z;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xFFFFFFFFu, s, o);
    if ((threadIdx.x & 31) == 0) atomicAdd(out, s);
}

inline unsigned blocks_for(size_t threads, unsigned per) {
    return static_cast<unsigned>((threads + per - 1) / per);
}

}  // namespace

cudaError_t launch_layernorm(const float* x, int rows, int D, int rpb, const float* shift,
                             const float* scale, int mod_ld, const void* w, const void* b,
                             float eps, void* out, cudaStream_t s, unsigned long long* launches) {
    if (rows <= 0) return cudaSuccess;
    // DLO_LN_WPR=1|2|4|8 forces the warps per row (tuning)
    static int forced = -1;
    if (forced < 0) {
        const char* e = std::getenv("DLO_LN_WPR");
        forced = e ? std::atoi(e) : 0;
    }
    // Two warps per row, more only for rows wider than 20 float4 per thread
    // (registers decide occupancy).  Measured on GB300, back to back: 2048 x
    // 1152 rows take 6.9 us with two warps per row against 9.0 / 11.6 / 10.5
    // with one / four / eight, 256 x 256 8.6 against 10.3-10.9, and 8192 or
    // 32760 x 5120 are fastest at two as well.
    const int n4 = D / 4;
    int wpr = 2;
    while (wpr < 8 && (n4 + 32 * wpr - 1) / (32 * wpr) > 20) wpr *= 2;
    if (forced == 1 || forced == 2 || forced == 4 || forced == 8) wpr = forced;
    if ((n4 + 32 * wpr - 1) / (32 * wpr) > (wpr == 1 ? 40 : 20)) return cudaErrorInvalidValue;
    const int v4 = (n4 + 32 * wpr - 1) / (32 * wpr);   // float4 per thread
    const unsigned g = static_cast<unsigned>((rows + 8 / wpr - 1) / (8 / wpr));
    const __nv_bfloat16* wb = static_cast<const __nv_bfloat16*>(w);
    const __nv_bfloat16* bb = static_cast<const __nv_bfloat16*>(b);
    __nv_bfloat16* o = static_cast<__nv_bfloat16*>(out);
    cudaError_t le_ = cudaErrorInvalidValue;
#define DLO_LN(V, W) \
    le_ = launch_k(layernorm_kernel<V, W>, g, 256, 0, s, x, rows, D, rpb, shift, scale, mod_ld, wb, bb, eps, o)
    if (wpr == 1) {
        if (v4 <= 2) DLO_LN(2, 1);
        else if (v4 <= 4) DLO_LN(4, 1);
        else if (v4 <= 8) DLO_LN(8, 1);
        else if (v4 <= 10) DLO_LN(10, 1);
        else if (v4 <= 16) DLO_LN(16, 1);
        else if (v4 <= 24) DLO_LN(24, 1);
        else if (v4 <= 32) DLO_LN(32, 1);
        else if (v4 <= 40) DLO_LN(40, 1);
        else return cudaErrorInvalidValue;
    } else {
#define DLO_LN_V(W)                   \
    if (v4 <= 1) DLO_LN(1, W);        \
    else if (v4 <= 2) DLO_LN(2, W);   \
    else if (v4 <= 3) DLO_LN(3, W);   \
    else if (v4 <= 5) DLO_LN(5, W);   \
    else if (v4 <= 10) DLO_LN(10, W); \
    else if (v4 <= 20) DLO_LN(20, W); \
    else return cudaErrorInvalidValue;
        if (wpr == 2) { DLO_LN_V(2) }
        else if (wpr == 4) { DLO_LN_V(4) }
        else { DLO_LN_V(8) }
#undef DLO_LN_V
    }
#undef DLO_LN
    ++*launches;
    return le_ != cudaSuccess ? le_ : cudaGetLastError();
}

cudaError_t launch_rmsnorm(void* x, int rows, int D, int ld, int col0, const void* w, float eps,
                           cudaStream_t s, unsigned long long* launches) {
    if (rows <= 0) return cudaSuccess;
    cudaError_t le_ = launch_k(rmsnorm_kernel, blocks_for(static_cast<size_t>(rows) * 32, 256), 256, 0, s, static_cast<__nv_bfloat16*>(x), rows, D, ld, col0, static_cast<const __nv_bfloat16*>(w),
        0, nullptr, eps);
    ++*launches;
    return le_ != cudaSuccess ? le_ : cudaGetLastError();
}

cudaError_t launch_rmsnorm2(void* x, int rows, int D, int ld, int col0a, const void* wa,
                            int col0b, const void* wb, float eps, cudaStream_t s,
                            unsigned long long* launches) {
    if (rows <= 0) return cudaSuccess;
    cudaError_t le_ = launch_k(rmsnorm_kernel, blocks_for(static_cast<size_t>(rows) * 64, 256), 256, 0, s, static_cast<__nv_bfloat16*>(x), rows, D, ld, col0a,
        static_cast<const __nv_bfloat16*>(wa), col0b, static_cast<const __nv_bfloat16*>(wb), eps);
    ++*launches;
    return le_ != cudaSuccess ? le_ : cudaGetLastError();
}

cudaError_t launch_adaln(const void* c, int B, int C, const void* W, const void* bias, int N,
                         float* m, cudaStream_t s, unsigned long long* launches, bool w_ready) {
    if (N <= 0 || B <= 0) return cudaSuccess;
    static int sms = 0;
    if (!sms) {
        int dev = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (sms <= 0) sms = 1;
    }
    // rows per warp: the fewest that keep the grid within one wave of two
    // 256-thread CTAs per SM
    const long long warps = 2LL * sms * 8;
    const int rows = N <= warps ? 1 : N <= 2 * warps ? 2 : N <= 3 * warps ? 3 : 4;
    const unsigned g = static_cast<unsigned>((N + 8 * rows - 1) / (8 * rows));
    const __nv_bfloat16* cb = static_cast<const __nv_bfloat16*>(c);
    const __nv_bfloat16* Wb = static_cast<const __nv_bfloat16*>(W);
    const __nv_bfloat16* bb = static_cast<const __nv_bfloat16*>(bias);
    cudaError_t le_ = cudaSuccess;
#define DLO_ADALN(BC, R)                                                                            \
    le_ = w_ready ? launch_k(adaln_kernel<BC, R, true>, g, 256, (BC) * ADALN_CCH * sizeof(float), s, cb, B, C, \
                             Wb, bb, N, m)                                                            \
                  : launch_k(adaln_kernel<BC, R, false>, g, 256, (BC) * ADALN_CCH * sizeof(float), s, cb, B, \
                             C, Wb, bb, N, m)
#define DLO_ADALN_R(BC)           \
    if (rows == 1) DLO_ADALN(BC, 1); \
    else if (rows == 2) DLO_ADALN(BC, 2); \
    else if (rows == 3) DLO_ADALN(BC, 3); \
    else DLO_ADALN(BC, 4)
    if (B <= 1) { DLO_ADALN_R(1); }
    else if (B <= 2) { DLO_ADALN_R(2); }
    else { DLO_ADALN_R(4); }
#undef DLO_ADALN_R
#undef DLO_ADALN
    ++*launches;
    return le_ != cudaSuccess ? le_ : cudaGetLastError();
}

cudaError_t launch_mod_add(const float* e, const void* table, int B, int n6d, float* m,
                           cudaStream_t s, unsigned long long* launches) {
    const size_t n = static_cast<size_t>(B) * n6d;
    if (!n) return cudaSuccess;
    cudaError_t le_ = launch_k(mod_add_kernel, blocks_for(n, 256), 256, 0, s, e, static_cast<const __nv_bfloat16*>(table),
                                                      B, n6d, m);
    ++*launches;
    return le_ != cudaSuccess ? le_ : cudaGetLastError();
}

cudaError_t launch_bf16_to_f32(const void* in, float* out, size_t n, cudaStream_t s,
                               unsigned long long* launches) {
    const size_t n8 = n / 8;
    if (!n8) return cudaSuccess;
    cudaError_t le_ = launch_k(bf16_to_f32_kernel, blocks_for(n8, 256), 256, 0, s, static_cast<const __nv_bfloat16*>(in),
                                                           out, n8);
    ++*launches;
    return le_ != cudaSuccess ? le_ : cudaGetLastError();
}

cudaError_t launch_f32_to_bf16(const float* in, void* out, size_t n, cudaStream_t s,
                               unsigned long long* launches) {
    const size_t n8 = n / 8;
    if (!n8) return cudaSuccess;
    cudaError_t le_ = launch_k(f32_to_bf16_kernel, blocks_for(n8, 256), 256, 0, s, in, static_cast<__nv_bfloat16*>(out),
                                                           n8);
    ++*launches;
    return le_ != cudaSuccess ? le_ : cudaGetLastError();
}

cudaError_t launch_quantize_e4m3(const void* x, int rows, int cols, int ld, void* q, float* scale,
                                 float* scratch, cudaStream_t s, unsigned long long* launches) {
    if (rows <= 0) return cudaSuccess;
    static int grid = 0;
    if (!grid) {
        int dev = 0, sms = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        grid = sms > 0 ? 4 * sms : 128;
        if (grid > kQuantScratch) grid = kQuantScratch;
    }
    const int c8 = cols / 8;
    const long long chunks = 1LL * rows * c8;
    long long need = (chunks + 255) / 256;
    const int g = static_cast<int>(need < grid ? (need > 0 ? need : 1) : grid);
    const __nv_bfloat16* xb = static_cast<const __nv_bfloat16*>(x);
    cudaError_t le_ = launch_k(amax_partial_kernel, g, 256, 0, s, xb, rows, c8, ld, scratch);
    if (le_ == cudaSuccess)
        le_ = launch_k(quant_e4m3_kernel, g, 256, 0, s, xb, rows, c8, ld, scratch, g, static_cast<uint8_t*>(q), scale);
    *launches += 2;
    return le_ != cudaSuccess ? le_ : cudaGetLastError();
}

cudaError_t launch_wait_selftest(int* err, cudaStream_t s, unsigned long long* launches) {
    cudaError_t le_ = launch_k(wait_selftest_kernel, 1, 32, 0, s, err);
    ++*launches;
    return le_ != cudaSuccess ? le_ : cudaGetLastError();
}

cudaError_t launch_gather(void* dst, const void* src, size_t bytes, cudaStream_t s,
                          unsigned long long* launches) {
    const size_t n16 = bytes / 16;
    if (!n16) return cudaSuccess;
    static int grid = 0;
    if (!grid) {
        int dev = 0, sms = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        grid = sms > 0 ? sms / 4 : 32;   // a quarter of the SMs
    }
    unsigned g = static_cast<unsigned>(grid);
    const size_t need = (n16 + 1023) / 1024;
    if (need < g) g = static_cast<unsigned>(need);
    gather_kernel<<<g, 1024, 0, s>>>(static_cast<uint4*>(dst), static_cast<const uint4*>(src),
                                     n16);
    ++*launches;
    return cudaGetLastError();
}

cudaError_t launch_checksum(const void* src, size_t bytes, unsigned long long* out, cudaStream_t s,
                            unsigned long long* launches) {
    const size_t n16 = bytes / 16;
    if (!n16) return cudaSuccess;
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    size_t g = static_cast<size_t>(sms > 0 ? sms : 1) * 8;
    const size_t need = (n16 + 255) / 256;
    if (need < g) g = need;
    cudaError_t le_ = launch_k(checksum_kernel, static_cast<unsigned>(g), 256, 0, s, static_cast<const uint4*>(src), n16, out);
    ++*launches;
    return le_ != cudaSuccess ? le_ : cudaGetLastError();
}

}  // namespace dlo
