// Internal declarations shared by the host runtime and the kernel files.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <cstddef>
#include <cstdint>
#include <string>
#include <vector>

#include "dlo.h"

namespace dlo {

// Programmatic dependent launch: on unless DLO_PDL=0 (diagnosis).
bool pdl_enabled();

// Launch `kernel` on `s` allowing programmatic stream serialisation (the
// kernel must run pdl_wait() before touching global memory).
template <typename... KArgs, typename... Args>
cudaError_t launch_k(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                     Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = pdl_enabled() ? 1 : 0;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// ------------------------------------------------------------------ layout

// Linear weights stored as E4M3 codes (W8A16 or W8A8).
inline bool e4m3_weights(int wdtype) { return wdtype == DLO_W_E4M3 || wdtype == DLO_W_E4M3_A8; }

struct Entry {
    std::string name;
    size_t offset = 0;
    size_t bytes = 0;
    int dtype = DLO_DT_BF16;
    int ndim = 1;
    long long shape[2] = {0, 0};
    int source = 1;
};

// Validates the description; returns DLO_OK or an error with a message.
dlo_status validate_desc(const dlo_desc* d, std::string* msg);
// Builds the flat block layout (groups start 256-B aligned; members of a
// group are contiguous).  Returns total bytes (multiple of 256).
size_t build_layout(const dlo_desc& d, std::vector<Entry>* out);
// Validates an ordered list of n container descriptions: each valid, the
// shared fields equal, bytes blocks alone.  *stack (may be NULL) receives the
// stack-wide description: container 0's fields, n_blocks = all blocks, the
// text fields of the video containers.
dlo_status validate_stack(const dlo_desc* ds, int n, dlo_desc* stack, std::string* msg);
int find_entry(const std::vector<Entry>& L, const char* name);

// Device workspace carve-up for max_batch x max_tokens activations.
struct Workspace {
    size_t x = 0;        // fp32 [BN, D]   hidden state
    size_t h = 0;        // bf16 [BN, D]   norm output
    size_t big = 0;      // bf16 [BN, max(3D, F)]  qkv, then FFN hidden
    size_t a = 0;        // bf16 [BN, D]   attention output
    size_t q2 = 0;       // bf16 [BN, D]   cross-attention q (video)
    size_t kv2 = 0;      // bf16 [B*L, 2D] cross-attention k|v (video)
    size_t mod = 0;      // fp32 [B, 6D]   modulation
    size_t in_x = 0;     // bf16 [BN, D]   staging of host inputs (forward_host)
    size_t in_cond = 0;  // cond staging (forward_host)
    size_t in_ctx = 0;   // bf16 [B*L, Dt] (forward_host)
    size_t qa = 0;       // W8A8: E4M3 codes of the current linear's input
    size_t qs = 0;       // W8A8: kQuantScratch partial maxima, then the scale
    size_t wide = 0;     // W8A16: bf16 copy of the current linear's weights
    size_t wide_bytes = 0;   // its size (0: no such buffer)
    size_t gsync = 0;    // W8A16: the widening GEMM's grid-barrier counter
    size_t err = 0;      // int[64] kernels' error words
    size_t total = 0;
};
// wide_min: bytes of the W8A16 widened-weight buffer at least (a stack
// whose containers differ in weight type).
Workspace plan_workspace(const dlo_desc& d, size_t wide_min = 0);
// Bytes of the W8A16 widened-weight buffer of one block type (its largest
// linear in bf16), 0 unless its weights are W8A16.
size_t widen_buffer_bytes(const dlo_desc& d);
// One workspace that serves every container of a stack.
Workspace plan_workspace_stack(const dlo_desc* ds, int n);

// ------------------------------------------------------------------ host math

uint16_t f32_to_bf16_rne(float f);
uint8_t f32_to_e4m3_rne_sat(float v);

// ------------------------------------------------------------------ kernel launchers
// All return cudaSuccess or the launch error; arguments are validated by the
// callers.  Each increments *launches by the kernels it launched.

struct GemmParams {
    const void* A = nullptr;      // bf16 [M, K]
    const void* W = nullptr;      // [N, K] bf16 or e4m3
    int w_dtype = DLO_DT_BF16;
    const float* scales = nullptr;
    int scale_seg = 0;
    int a_dtype = DLO_DT_BF16;        // DLO_DT_E4M3: A holds E4M3 codes [M, K] (W8A8)
    const float* a_scale = nullptr;   // W8A8: device fp32 activation scale
    const void* bias = nullptr;   // bf16 [N]
    int M = 0, N = 0, K = 0;
    int epi = DLO_EPI_BIAS;
    void* out = nullptr;
    int ldo = 0;
    const float* gate = nullptr;
    int gate_ld = 0;
    int rows_per_batch = 1;
    int* err = nullptr;
    // W is not written by the kernel before this one in the stream (block
    // weights staged, and waited for, before the block's first kernel): the
    // producer then loads the first stages' weight tiles before the
    // programmatic-launch wait, overlapping the predecessor's tail.
    bool w_ready = false;
    // W8A16 dequantised inside the GEMM: E4M3 codes [N, K] (16-B aligned,
    // N*K a multiple of 16) that the kernel widens into W (a bf16 [N, K]
    // buffer it then multiplies, w_dtype bf16, scales applied as usual) before
    // its mainloop, with w_sync a device counter for its grid barrier.
    const void* w_codes = nullptr;
    unsigned* w_sync = nullptr;
};
cudaError_t launch_gemm(const GemmParams& p, cudaStream_t s, unsigned long long* launches);
// E4M3 codes [n] -> bf16 [n], exactly (the codes' values; a per-tensor scale
// stays with the GEMM's epilogue).  codes and out 16-byte aligned.
cudaError_t launch_widen_e4m3(const void* codes, size_t n, void* out, cudaStream_t s,
                              unsigned long long* launches);
int gemm_num_sms();

// Unit-op plumbing shared by the C ABI's op entry points.  op_fail stores the
// message that dlo_last_error(NULL) returns and passes the status through;
// op_result turns a launch error into DLO_ECUDA the same way.
dlo_status op_fail(dlo_status st, const std::string& msg);
dlo_status op_result(cudaError_t e);
// The argument checks of the GEMM ops and their GemmParams (p->err left NULL).
dlo_status op_gemm_params(const void* A, const void* W, int w_dtype, const float* scales, int scale_seg,
                          const void* bias, int M, int N, int K, int epilogue, void* out, int ldo,
                          const float* gate, int gate_ld, int rows_per_batch, int a_dtype,
                          const float* a_scale, GemmParams* p);
// launch_gemm, counted with the unit ops' launches, through op_result.
dlo_status op_launch_gemm(const GemmParams& p, cudaStream_t s);

// cuTensorMapEncodeTiled, resolved once through the runtime's driver entry
// point (no link-time dependency on libcuda) and wrapped by a table of
// already-encoded maps keyed by every argument; NULL if unavailable.
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn tensor_map_encoder();

// Attention on the tcgen05 kernel (head dims: multiples of 8 up to 128).
// err: device error word or NULL.
cudaError_t launch_attention(const void* Q, const void* K, const void* V, void* O, int batch,
                             int heads, int hd, int nq, int nk, int ldq, int ldk, int ldv, int ldo,
                             int* err, cudaStream_t s, unsigned long long* launches);
bool attention_tc_supported(int hd);
cudaError_t launch_attention_tc(const void* Q, const void* K, const void* V, void* O, int batch,
                                int heads, int hd, int nq, int nk, int ldq, int ldk, int ldv,
                                int ldo, int* err, cudaStream_t s, unsigned long long* launches);

cudaError_t launch_layernorm(const float* x, int rows, int D, int rpb, const float* shift,
                             const float* scale, int mod_ld, const void* w, const void* b,
                             float eps, void* out, cudaStream_t s, unsigned long long* launches);
cudaError_t launch_rmsnorm(void* x, int rows, int D, int ld, int col0, const void* w, float eps,
                           cudaStream_t s, unsigned long long* launches);
// Two segments of one row set in one launch (q and k of the same rows).
cudaError_t launch_rmsnorm2(void* x, int rows, int D, int ld, int col0a, const void* wa,
                            int col0b, const void* wb, float eps, cudaStream_t s,
                            unsigned long long* launches);
// w_ready: W is not written by the kernel before this one in the stream (the
// first W loads may then start before the programmatic-launch wait).
cudaError_t launch_adaln(const void* c, int B, int C, const void* W, const void* bias, int N,
                         float* m, cudaStream_t s, unsigned long long* launches, bool w_ready = false);
cudaError_t launch_mod_add(const float* e, const void* table, int B, int n6d, float* m,
                           cudaStream_t s, unsigned long long* launches);
cudaError_t launch_bf16_to_f32(const void* in, float* out, size_t n, cudaStream_t s,
                               unsigned long long* launches);
cudaError_t launch_f32_to_bf16(const float* in, void* out, size_t n, cudaStream_t s,
                               unsigned long long* launches);
cudaError_t launch_gather(void* dst, const void* src, size_t bytes, cudaStream_t s,
                          unsigned long long* launches);
// One thread waits on an mbarrier nothing completes; when the bounded wait
// runs out it sets *err = 1 (device) and the kernel exits.
cudaError_t launch_wait_selftest(int* err, cudaStream_t s, unsigned long long* launches);
// Dynamic per-tensor E4M3 quantisation of a bf16 [rows, cols] activation
// (row stride ld, cols % 8 == 0, 16-B aligned rows) into contiguous codes q
// [rows, cols] and the fp32 scale *scale (device); scratch holds
// kQuantScratch floats of partial maxima.
constexpr int kQuantScratch = DLO_QUANT_SCRATCH;
cudaError_t launch_quantize_e4m3(const void* x, int rows, int cols, int ld, void* q, float* scale,
                                 float* scratch, cudaStream_t s, unsigned long long* launches);
// *out += sum of the 64-bit words of src (bytes % 16 == 0), mod 2^64.
cudaError_t launch_checksum(const void* src, size_t bytes, unsigned long long* out, cudaStream_t s,
                            unsigned long long* launches);

}  // namespace dlo
