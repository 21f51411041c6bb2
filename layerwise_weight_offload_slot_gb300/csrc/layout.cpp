// Flat block layout (one table for every block of a stack), host packing,
// bf16 rounding and the per-tensor E4M3 quantiser.
//
// "CPU Offloading for Diffusion Models", Layerwise (Blockwise) Offloading,
// How It Works: block parameters are retained as flattened tensors in pinned
// host memory and re-materialised from them.  "Distributed Layerwise
// Offload", Registered runtime-cache transfer: each tensor has a fixed offset
// in the flattened rotating device buffer.  Here every tensor group starts
// 256-byte aligned so that the same offsets serve the host block, both device
// slots and the resident buffers, and every TMA descriptor base is aligned.
#include <algorithm>
#include <cmath>
#include <cstring>
#include <string>
#include <vector>

#include "internal.h"

namespace dlo {

static size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

dlo_status validate_desc(const dlo_desc* d, std::string* msg) {
    auto fail = [&](dlo_status st, const char* m) {
        if (msg) *msg = m;
        return st;
    };
    if (!d) return fail(DLO_EINVAL, "desc is NULL");
    if (d->abi_version != DLO_ABI_VERSION) return fail(DLO_EINVAL, "abi_version mismatch");
    if (d->block_kind != DLO_BLOCK_DIT && d->block_kind != DLO_BLOCK_VIDEO &&
        d->block_kind != DLO_BLOCK_BYTES)
        return fail(DLO_EINVAL, "unknown block_kind");
    if (d->block_kind == DLO_BLOCK_BYTES) {
        if (d->n_blocks < 1) return fail(DLO_EINVAL, "n_blocks < 1");
        if (d->bytes_block == 0 || d->bytes_block % 256 != 0)
            return fail(DLO_EINVAL, "bytes_block must be a positive multiple of 256");
        if (d->staging != DLO_STAGE_MEMCPY && d->staging != DLO_STAGE_GATHER &&
            d->staging != DLO_STAGE_PER_TENSOR)
            return fail(DLO_EINVAL, "unknown staging");
        return DLO_OK;
    }
    if (d->wdtype != DLO_W_BF16 && !e4m3_weights(d->wdtype)) return fail(DLO_EINVAL, "unknown wdtype");
    if (d->n_blocks < 1) return fail(DLO_EINVAL, "n_blocks < 1");
    if (d->heads < 1 || d->head_dim < 8 || d->hidden != d->heads * d->head_dim)
        return fail(DLO_EINVAL, "hidden must equal heads * head_dim");
    if (d->hidden % 16 != 0) return fail(DLO_EINVAL, "hidden % 16 != 0");
    if (d->head_dim % 8 != 0 || d->head_dim > 128) return fail(DLO_EINVAL, "head_dim must be a multiple of 8, <= 128");
    if (d->ffn < 16 || d->ffn % 16 != 0) return fail(DLO_EINVAL, "ffn % 16 != 0");
    if (d->max_batch < 1 || d->max_tokens < 1) return fail(DLO_EINVAL, "max_batch/max_tokens < 1");
    if (!(d->eps > 0.0f)) return fail(DLO_EINVAL, "eps <= 0");
    if (d->staging != DLO_STAGE_MEMCPY && d->staging != DLO_STAGE_GATHER &&
        d->staging != DLO_STAGE_PER_TENSOR)
        return fail(DLO_EINVAL, "unknown staging");
    if (d->block_kind == DLO_BLOCK_DIT) {
        if (d->cond_dim < 8 || d->cond_dim % 16 != 0) return fail(DLO_EINVAL, "cond_dim % 16 != 0");
        if (e4m3_weights(d->wdtype))
            return fail(DLO_EUNSUPPORTED, "E4M3 weights are implemented for video blocks only");
    } else {
        if (d->text_dim < 16 || d->text_dim % 16 != 0) return fail(DLO_EINVAL, "text_dim % 16 != 0");
        if (d->max_text_tokens < 1) return fail(DLO_EINVAL, "max_text_tokens < 1");
    }
    const long long bn = 1LL * d->max_batch * d->max_tokens;
    if (bn > (1LL << 30) / 4) return fail(DLO_EINVAL, "max_batch * max_tokens too large");
    return DLO_OK;
}

dlo_status validate_stack(const dlo_desc* ds, int n, dlo_desc* stack, std::string* msg) {
    auto fail = [&](dlo_status st, const char* m) {
        if (msg) *msg = m;
        return st;
    };
    if (!ds) return fail(DLO_EINVAL, "descs is NULL");
    if (n < 1 || n > DLO_MAX_CONTAINERS) return fail(DLO_EINVAL, "n_containers out of range");
    long long total = 0;
    int video = -1;
    for (int i = 0; i < n; ++i) {
        dlo_status st = validate_desc(&ds[i], msg);
        if (st != DLO_OK) return st;
        const dlo_desc& a = ds[i];
        const dlo_desc& z = ds[0];
        if (n > 1 && a.block_kind == DLO_BLOCK_BYTES)
            return fail(DLO_EINVAL, "bytes blocks cannot share a stack with other containers");
        if (a.hidden != z.hidden || a.max_batch != z.max_batch || a.max_tokens != z.max_tokens ||
            a.eps != z.eps || a.staging != z.staging || a.register_budget_bytes != z.register_budget_bytes)
            return fail(DLO_EINVAL,
                        "containers must share hidden, max_batch, max_tokens, eps, staging and "
                        "register_budget_bytes");
        if (a.block_kind == DLO_BLOCK_VIDEO) {
            if (video >= 0 && (a.text_dim != ds[video].text_dim ||
                               a.max_text_tokens != ds[video].max_text_tokens))
                return fail(DLO_EINVAL, "video containers must share text_dim and max_text_tokens");
            if (video < 0) video = i;
        }
        total += a.n_blocks;
    }
    if (total > (1LL << 24)) return fail(DLO_EINVAL, "too many blocks");
    if (stack) {
        *stack = ds[0];
        stack->n_blocks = static_cast<int>(total);
        if (video >= 0) {
            stack->text_dim = ds[video].text_dim;
            stack->max_text_tokens = ds[video].max_text_tokens;
        }
    }
    return DLO_OK;
}

Workspace plan_workspace_stack(const dlo_desc* ds, int n) {
    // one carve-up that serves every container: the widest FFN, the
    // cross-attention buffers when any container is a video one, and the
    // largest W8A16 widened-weight buffer
    dlo_desc u = ds[0];
    size_t wide = 0;
    for (int i = 0; i < n; ++i) {
        wide = std::max(wide, widen_buffer_bytes(ds[i]));
        u.ffn = std::max(u.ffn, ds[i].ffn);
        u.cond_dim = std::max(u.cond_dim, ds[i].cond_dim);
        if (ds[i].wdtype == DLO_W_E4M3_A8) u.wdtype = DLO_W_E4M3_A8;
        if (ds[i].block_kind == DLO_BLOCK_VIDEO) {
            u.block_kind = DLO_BLOCK_VIDEO;
            u.text_dim = ds[i].text_dim;
            u.max_text_tokens = ds[i].max_text_tokens;
        }
    }
    return plan_workspace(u, wide);
}

size_t widen_buffer_bytes(const dlo_desc& d) {
    if (d.wdtype != DLO_W_E4M3 || d.block_kind == DLO_BLOCK_BYTES) return 0;
    const size_t D = d.hidden, F = d.ffn;
    size_t nk = std::max(3 * D * D, F * D);   // qkv; fc1 and fc2
    if (d.block_kind == DLO_BLOCK_VIDEO) nk = std::max(nk, 2 * D * static_cast<size_t>(d.text_dim));   // cross k|v
    return nk * 2;
}

namespace {
struct Builder {
    std::vector<Entry>* out;
    size_t cur = 0;
    void group() { cur = align_up(cur, 256); }
    void add(const char* name, int dtype, long long s0, long long s1 = -1, int source = 1) {
        Entry e;
        e.name = name;
        e.dtype = dtype;
        e.ndim = s1 < 0 ? 1 : 2;
        e.shape[0] = s0;
        e.shape[1] = s1 < 0 ? 0 : s1;
        size_t n = static_cast<size_t>(s0) * static_cast<size_t>(s1 < 0 ? 1 : s1);
        size_t es = dtype == DLO_DT_BF16 ? 2 : (dtype == DLO_DT_E4M3 || dtype == DLO_DT_U8) ? 1 : 4;
        e.offset = cur;
        e.bytes = n * es;
        e.source = source;
        cur += e.bytes;
        out->push_back(e);
    }
};
}  // namespace

size_t build_layout(const dlo_desc& d, std::vector<Entry>* out) {
    out->clear();
    Builder b{out};
    if (d.block_kind == DLO_BLOCK_BYTES) {
        b.group(); b.add("bytes", DLO_DT_U8, static_cast<long long>(d.bytes_block));
        b.group();
        return b.cur;
    }
    const long long D = d.hidden, F = d.ffn;
    const int W = e4m3_weights(d.wdtype) ? DLO_DT_E4M3 : DLO_DT_BF16;
    const int H = DLO_DT_BF16;
    if (d.block_kind == DLO_BLOCK_DIT) {
        const long long C = d.cond_dim;
        b.group(); b.add("adaLN.weight", H, 6 * D, C);
        b.group(); b.add("adaLN.bias", H, 6 * D);
        b.group(); b.add("attn.qkv.weight", W, 3 * D, D);
        b.group(); b.add("attn.qkv.bias", H, 3 * D);
        b.group(); b.add("attn.proj.weight", W, D, D);
        b.group(); b.add("attn.proj.bias", H, D);
        b.group(); b.add("mlp.fc1.weight", W, F, D);
        b.group(); b.add("mlp.fc1.bias", H, F);
        b.group(); b.add("mlp.fc2.weight", W, D, F);
        b.group(); b.add("mlp.fc2.bias", H, D);
    } else {
        const long long Dt = d.text_dim;
        b.group(); b.add("modulation", H, 6, D);
        // q, k, v weights and biases are contiguous groups: one fused GEMM
        b.group(); b.add("self_attn.q.weight", W, D, D);
        b.add("self_attn.k.weight", W, D, D);
        b.add("self_attn.v.weight", W, D, D);
        b.group(); b.add("self_attn.q.bias", H, D);
        b.add("self_attn.k.bias", H, D);
        b.add("self_attn.v.bias", H, D);
        b.group(); b.add("self_attn.o.weight", W, D, D);
        b.group(); b.add("self_attn.o.bias", H, D);
        b.group(); b.add("self_attn.norm_q.weight", H, D);
        b.group(); b.add("self_attn.norm_k.weight", H, D);
        b.group(); b.add("norm_cross.weight", H, D);
        b.group(); b.add("norm_cross.bias", H, D);
        b.group(); b.add("cross_attn.q.weight", W, D, D);
        b.group(); b.add("cross_attn.q.bias", H, D);
        b.group(); b.add("cross_attn.k.weight", W, D, Dt);
        b.add("cross_attn.v.weight", W, D, Dt);
        b.group(); b.add("cross_attn.k.bias", H, D);
        b.add("cross_attn.v.bias", H, D);
        b.group(); b.add("cross_attn.o.weight", W, D, D);
        b.group(); b.add("cross_attn.o.bias", H, D);
        b.group(); b.add("cross_attn.norm_q.weight", H, D);
        b.group(); b.add("cross_attn.norm_k.weight", H, D);
        b.group(); b.add("ffn.fc1.weight", W, F, D);
        b.group(); b.add("ffn.fc1.bias", H, F);
        b.group(); b.add("ffn.fc2.weight", W, D, F);
        b.group(); b.add("ffn.fc2.bias", H, D);
        if (e4m3_weights(d.wdtype)) {
            // one fp32 scale per linear: self q,k,v,o, cross q,k,v,o, fc1, fc2
            b.group(); b.add("linear_scales", DLO_DT_F32, 16, -1, 0);
        }
    }
    b.group();
    return b.cur;
}

int find_entry(const std::vector<Entry>& L, const char* name) {
    for (size_t i = 0; i < L.size(); ++i)
        if (L[i].name == name) return static_cast<int>(i);
    return -1;
}

Workspace plan_workspace(const dlo_desc& d, size_t wide_min) {
    Workspace w;
    if (d.block_kind == DLO_BLOCK_BYTES) {
        // error words, then the per-block checksums of dlo_forward_host
        w.err = 0;
        w.in_x = 256;
        w.total = align_up(256 + static_cast<size_t>(d.n_blocks) * 8, 256);
        return w;
    }
    const size_t BN = static_cast<size_t>(d.max_batch) * d.max_tokens;
    const size_t D = d.hidden, F = d.ffn;
    size_t cur = 0;
    auto take = [&](size_t bytes) {
        cur = align_up(cur, 256);
        size_t off = cur;
        cur += bytes;
        return off;
    };
    w.x = take(BN * D * 4);
    w.h = take(BN * D * 2);
    w.big = take(BN * std::max(3 * D, F) * 2);
    w.a = take(BN * D * 2);
    if (d.block_kind == DLO_BLOCK_VIDEO) {
        const size_t BL = static_cast<size_t>(d.max_batch) * d.max_text_tokens;
        w.q2 = take(BN * D * 2);
        w.kv2 = take(BL * 2 * D * 2);
        w.in_ctx = take(BL * d.text_dim * 2);
        w.in_cond = take(static_cast<size_t>(d.max_batch) * 6 * D * 4);
    } else {
        w.in_cond = take(static_cast<size_t>(d.max_batch) * d.cond_dim * 2);
    }
    w.mod = take(static_cast<size_t>(d.max_batch) * 6 * D * 4);
    w.in_x = take(BN * D * 2);
    if (d.wdtype == DLO_W_E4M3_A8) {
        // codes of the widest linear input: fc2's [BN, F], or the text context
        const size_t BL = static_cast<size_t>(d.max_batch) * d.max_text_tokens;
        w.qa = take(std::max(BN * std::max(D, F), BL * static_cast<size_t>(d.text_dim)));
        w.qs = take((kQuantScratch + 64) * sizeof(float));
    }
    w.wide_bytes = std::max(widen_buffer_bytes(d), wide_min);
    if (w.wide_bytes) {
        w.wide = take(w.wide_bytes);
        w.gsync = take(256);
    }
    w.err = take(64 * sizeof(int));
    w.total = align_up(cur, 256);
    return w;
}

// Round to nearest even from the fp32 bit pattern; NaN stays a quiet NaN.
uint16_t f32_to_bf16_rne(float f) {
    uint32_t u;
    std::memcpy(&u, &f, 4);
    if ((u & 0x7FFFFFFFu) > 0x7F800000u) return static_cast<uint16_t>((u >> 16) | 0x40u);
    const uint32_t lsb = (u >> 16) & 1u;
    u += 0x7FFFu + lsb;
    return static_cast<uint16_t>(u >> 16);
}

// E4M3 of a finite fp32 value: integer rounding of the fp32 significand at the
// E4M3 quantum of the value's binade (2^(E-3), E >= -6), ties to even,
// saturating to the largest finite magnitude 448 (code 0x7E).
uint8_t f32_to_e4m3_rne_sat(float v) {
    uint32_t u;
    std::memcpy(&u, &v, 4);
    const uint8_t sign = static_cast<uint8_t>((u >> 24) & 0x80u);
    const uint32_t biased = (u >> 23) & 0xFFu;
    if (biased == 0xFF) return sign | 0x7E;            // inf/NaN input: saturate
    if (biased == 0) return sign;                       // fp32 zero/subnormal -> 0
    const int exp = static_cast<int>(biased) - 127;     // value = m24 * 2^(exp-23)
    const uint32_t m24 = (u & 0x7FFFFFu) | 0x800000u;
    if (exp >= 9) return sign | 0x7E;                   // >= 512
    int E = exp < -6 ? -6 : exp;                        // target binade exponent
    const int shift = E - exp + 20;                     // m24 * 2^(exp-23) / 2^(E-3)
    uint32_t r;
    if (shift >= 32) {
        r = 0;
    } else {
        r = m24 >> shift;
        const uint32_t rem = m24 & ((1u << shift) - 1u);
        const uint32_t half = 1u << (shift - 1);
        if (rem > half || (rem == half && (r & 1u))) ++r;
    }
    uint32_t code;
    if (r >= 16) {          // rounded up into the next binade
        E += 1;
        r = 8;
    }
    if (r < 8) {
        code = r;           // subnormal (E == -6)
    } else {
        code = (static_cast<uint32_t>(E + 7) << 3) | (r - 8);
    }
    if (code > 0x7E) code = 0x7E;
    return static_cast<uint8_t>(sign | code);
}

}  // namespace dlo

using namespace dlo;

extern "C" size_t dlo_block_bytes(const dlo_desc* desc) {
    if (validate_desc(desc, nullptr) != DLO_OK) return 0;
    std::vector<Entry> L;
    return build_layout(*desc, &L);
}

extern "C" dlo_status dlo_block_layout(const dlo_desc* desc, dlo_tensor_info* out, int cap,
                                       int* count) {
    dlo_status st = validate_desc(desc, nullptr);
    if (st != DLO_OK) return st;
    std::vector<Entry> L;
    build_layout(*desc, &L);
    if (count) *count = static_cast<int>(L.size());
    if (!out) return DLO_OK;
    if (cap < static_cast<int>(L.size())) return DLO_ENOMEM;
    for (size_t i = 0; i < L.size(); ++i) {
        dlo_tensor_info& t = out[i];
        std::memset(&t, 0, sizeof(t));
        std::strncpy(t.name, L[i].name.c_str(), sizeof(t.name) - 1);
        t.offset = L[i].offset;
        t.bytes = L[i].bytes;
        t.dtype = L[i].dtype;
        t.ndim = L[i].ndim;
        t.shape[0] = L[i].shape[0];
        t.shape[1] = L[i].shape[1];
        t.source = L[i].source;
    }
    return DLO_OK;
}

extern "C" size_t dlo_workspace_bytes(const dlo_desc* desc) {
    if (validate_desc(desc, nullptr) != DLO_OK) return 0;
    return plan_workspace(*desc).total;
}

extern "C" size_t dlo_workspace_bytes_multi(const dlo_desc* descs, int n_containers) {
    if (validate_stack(descs, n_containers, nullptr, nullptr) != DLO_OK) return 0;
    return plan_workspace_stack(descs, n_containers).total;
}

extern "C" dlo_status dlo_quantize_e4m3(const float* w, size_t n, uint8_t* codes, float* scale) {
    if ((n && (!w || !codes)) || !scale) return DLO_EINVAL;
    float amax = 0.0f;
    for (size_t i = 0; i < n; ++i) {
        const float a = std::fabs(w[i]);
        if (!(a <= amax)) amax = a;      // also propagates NaN
    }
    if (!std::isfinite(amax)) return DLO_EINVAL;
    volatile float s = amax == 0.0f ? 1.0f : amax / 448.0f;
    const float sv = s;
    for (size_t i = 0; i < n; ++i) {
        volatile float v = w[i] / sv;
        codes[i] = f32_to_e4m3_rne_sat(v);
    }
    *scale = sv;
    return DLO_OK;
}

extern "C" dlo_status dlo_pack_block(const dlo_desc* desc, const float* const* tensors,
                                     int n_tensors, void* flat, size_t flat_bytes) {
    dlo_status st = validate_desc(desc, nullptr);
    if (st != DLO_OK) return st;
    std::vector<Entry> L;
    const size_t total = build_layout(*desc, &L);
    if (!tensors || !flat || n_tensors != static_cast<int>(L.size())) return DLO_EINVAL;
    if (flat_bytes < total) return DLO_ENOMEM;
    for (size_t i = 0; i < L.size(); ++i)
        if (L[i].source && !tensors[i]) return DLO_EINVAL;
    uint8_t* base = static_cast<uint8_t*>(flat);
    std::memset(base, 0, total);
    std::vector<float> scales;
    for (size_t i = 0; i < L.size(); ++i) {
        const Entry& e = L[i];
        if (!e.source) continue;
        const size_t n = static_cast<size_t>(e.shape[0]) * (e.ndim == 2 ? e.shape[1] : 1);
        const float* src = tensors[i];
        if (e.dtype == DLO_DT_BF16) {
            uint16_t* dst = reinterpret_cast<uint16_t*>(base + e.offset);
            for (size_t j = 0; j < n; ++j) dst[j] = f32_to_bf16_rne(src[j]);
        } else if (e.dtype == DLO_DT_U8) {
            return DLO_EINVAL;   // opaque byte blocks are written by the caller, not packed
        } else if (e.dtype == DLO_DT_E4M3) {
            float s = 1.0f;
            st = dlo_quantize_e4m3(src, n, base + e.offset, &s);
            if (st != DLO_OK) return st;
            scales.push_back(s);
        } else {
            std::memcpy(base + e.offset, src, n * 4);
        }
    }
    const int si = find_entry(L, "linear_scales");
    if (si >= 0) {
        float* dst = reinterpret_cast<float*>(base + L[si].offset);
        for (size_t j = 0; j < scales.size() && j < 16; ++j) dst[j] = scales[j];
    }
    return DLO_OK;
}
