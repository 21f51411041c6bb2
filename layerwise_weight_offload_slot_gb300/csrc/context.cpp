// Host runtime of the layerwise offload: context lifecycle, host block
// registration with all-or-nothing rollback, resident leading blocks,
// priming, the event-ordered two-slot circular prefetch, block orchestration,
// timing/overlap accounting and the C ABI.
//
// Sources: "CPU Offloading for Diffusion Models", Layerwise (Blockwise)
// Offloading (How It Works, Execution Flow table); "Distributed Layerwise
// Offload" (Startup and runtime sequence, Host backing and transfer
// composition, Failure and lifecycle boundaries, Registered runtime-cache
// transfer); "CPU Offloading" (Shared lifecycle, Cross-strategy invariants).
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <chrono>
#include <condition_variable>
#include <mutex>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <deque>
#include <memory>
#include <string>
#include <thread>
#include <vector>

#include "internal.h"

using namespace dlo;

namespace {

thread_local std::string g_create_error;
std::atomic<int> g_fail_register_nth{0};

enum State { kCreated = 0, kRegistered = 1, kBroken = 9 };

struct TimedExec {
    cudaEvent_t copy0, copy1, wait0, comp0, comp1;
};

struct TimedKernel {
    int cls;
    cudaEvent_t a, b;
    double flops, bytes;
};

struct Offsets {
    // DiT
    size_t ada_w, ada_b, qkv_w, qkv_b, proj_w, proj_b, fc1_w, fc1_b, fc2_w, fc2_b;
    // video
    size_t mod, sq_w, sq_b, so_w, so_b, snq, snk, ncw, ncb, cq_w, cq_b, ck_w, ck_b, co_w, co_b, cnq,
        cnk, scales;
    bool has_scales;
};

// One ordered block container: a run of blocks that share one description
// and so one flat layout.  A stack is one container or several executed in
// order as a single list of blocks ("CPU Offloading for Diffusion Models",
// Layerwise Offloading: models with multiple block types), all streamed
// through the same two slots, sized for the largest block.
struct Container {
    dlo_desc d{};
    std::vector<Entry> L;
    size_t block_bytes = 0;
    Offsets off{};
    int first = 0;
};

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// A few host threads that split one memcpy between them (the pack of a
// pageable block into a pinned host staging slot).
class CopyPool {
  public:
    explicit CopyPool(int n) {
        for (int i = 0; i < n; ++i) threads_.emplace_back([this, i] { loop(i); });
    }
    ~CopyPool() {
        {
            std::lock_guard<std::mutex> g(mu_);
            stop_ = true;
        }
        cv_.notify_all();
        for (auto& t : threads_) t.join();
    }
    void copy(void* dst, const void* src, size_t bytes) {
        const int n = static_cast<int>(threads_.size());
        std::unique_lock<std::mutex> g(mu_);
        dst_ = static_cast<uint8_t*>(dst);
        src_ = static_cast<const uint8_t*>(src);
        bytes_ = bytes;
        pending_ = n;
        ++gen_;
        cv_.notify_all();
        done_cv_.wait(g, [&] { return pending_ == 0; });
    }

  private:
    void loop(int i) {
        unsigned long long seen = 0;
        for (;;) {
            uint8_t* d;
            const uint8_t* s;
            size_t b;
            {
                std::unique_lock<std::mutex> g(mu_);
                cv_.wait(g, [&] { return stop_ || gen_ != seen; });
                if (stop_) return;
                seen = gen_;
                d = dst_;
                s = src_;
                b = bytes_;
            }
            const int n = static_cast<int>(threads_.size());
            const size_t chunk = (b / n + 4095) / 4096 * 4096;
            const size_t lo = std::min(b, chunk * i), hi = std::min(b, lo + chunk);
            if (hi > lo) std::memcpy(d + lo, s + lo, hi - lo);
            {
                std::lock_guard<std::mutex> g(mu_);
                if (--pending_ == 0) done_cv_.notify_all();
            }
        }
    }
    std::vector<std::thread> threads_;
    std::mutex mu_;
    std::condition_variable cv_, done_cv_;
    uint8_t* dst_ = nullptr;
    const uint8_t* src_ = nullptr;
    size_t bytes_ = 0;
    int pending_ = 0;
    unsigned long long gen_ = 0;
    bool stop_ = false;
};

// Packs pageable host blocks into the two pinned host staging slots on a
// thread of its own, so that the pack of one staging overlaps the
// host-to-device copy of the one before ("Distributed Layerwise Offload",
// Host backing and transfer composition: two bounded pinned host-staging
// slots).  Staging n uses host slot n % 2; its pack may start once the copy
// of staging n - 2, the slot's previous reader, has finished.  The copy
// stream learns that a pack is done from a host function that waits for it
// (wait_packed) and reports each finished copy through another (copied).
// Host functions here call no CUDA API.
class HostPacker {
  public:
    explicit HostPacker(int threads) : pool_(threads), thread_([this] { loop(); }) {}
    ~HostPacker() {
        {
            std::lock_guard<std::mutex> g(mu_);
            stop_ = true;
        }
        cv_.notify_all();
        thread_.join();
    }
    // Queue the pack of staging n (stagings are submitted in order).
    void submit(unsigned long long n, void* dst, const void* src, size_t bytes) {
        {
            std::lock_guard<std::mutex> g(mu_);
            jobs_.push_back(Job{n, dst, src, bytes});
        }
        cv_.notify_all();
    }
    // Blocks until the pack of staging n is done.
    void wait_packed(unsigned long long n) {
        std::unique_lock<std::mutex> g(mu_);
        cv_.wait(g, [&] { return packed_ > n || stop_; });
    }
    // The copy of staging n has finished.
    void copied(unsigned long long n) {
        {
            std::lock_guard<std::mutex> g(mu_);
            copied_ = std::max(copied_, n + 1);
        }
        cv_.notify_all();
    }
    // Packs that had to wait for their host slot (the copy two stagings
    // earlier still running), for the statistics.
    unsigned long long slot_waits() {
        std::lock_guard<std::mutex> g(mu_);
        return slot_waits_;
    }

  private:
    struct Job {
        unsigned long long n;
        void* dst;
        const void* src;
        size_t bytes;
    };
    void loop() {
        for (;;) {
            Job j;
            {
                std::unique_lock<std::mutex> g(mu_);
                cv_.wait(g, [&] { return stop_ || !jobs_.empty(); });
                if (stop_ && jobs_.empty()) return;
                j = jobs_.front();
                jobs_.pop_front();
                // the host slot's previous reader is the copy of staging n - 2
                if (j.n >= 2 && copied_ < j.n - 1) {
                    ++slot_waits_;
                    cv_.wait(g, [&] { return stop_ || copied_ >= j.n - 1; });
                    if (stop_) return;
                }
            }
            pool_.copy(j.dst, j.src, j.bytes);
            {
                std::lock_guard<std::mutex> g(mu_);
                packed_ = j.n + 1;
            }
            cv_.notify_all();
        }
    }
    CopyPool pool_;
    std::mutex mu_;
    std::condition_variable cv_;
    std::deque<Job> jobs_;
    unsigned long long packed_ = 0, copied_ = 0, slot_waits_ = 0;
    bool stop_ = false;
    std::thread thread_;
};

// Host threads of one pack (the memcpy of a block into a pinned host slot):
// DLO_PACK_THREADS, else 12.
int pack_threads() {
    const char* e = std::getenv("DLO_PACK_THREADS");
    const int v = e ? std::atoi(e) : 0;
    return v >= 1 && v <= 64 ? v : 12;
}

// Rows from which a W8A16 linear is widened to bf16 before its GEMM
// (DLO_WIDEN_ROWS, read once; default 4096).  Below that the widening stays
// inside the GEMM's mainloop, where a separate pass over the weights would
// cost more than it saves.
int widen_rows() {
    static int v = -1;
    if (v < 0) {
        const char* e = std::getenv("DLO_WIDEN_ROWS");
        const long long r = e ? std::atoll(e) : 0;
        v = r >= 1 && r <= (1ll << 30) ? static_cast<int>(r) : 4096;
    }
    return v;
}

struct PackTicket {
    HostPacker* packer;
    unsigned long long n;
};

void CUDART_CB wait_packed_fn(void* arg) {
    PackTicket* t = static_cast<PackTicket*>(arg);
    t->packer->wait_packed(t->n);
    delete t;
}

void CUDART_CB copied_fn(void* arg) {
    PackTicket* t = static_cast<PackTicket*>(arg);
    t->packer->copied(t->n);
    delete t;
}

}  // namespace

struct dlo_ctx {
    dlo_desc d{};                 // stack-wide: shared fields, n_blocks = all blocks
    int device = 0;
    std::vector<Container> conts;
    std::vector<int> cont_of;     // block index -> container index
    size_t block_bytes = 0;       // largest block: what a slot must hold
    Workspace ws;
    uint8_t* slot[2] = {nullptr, nullptr};
    size_t slot_bytes = 0;
    uint8_t* wsp = nullptr;
    cudaStream_t cs = nullptr;   // compute
    cudaStream_t xs = nullptr;   // copy
    cudaEvent_t copy_done[2] = {nullptr, nullptr};
    cudaEvent_t compute_done[2] = {nullptr, nullptr};
    cudaEvent_t resident_ev = nullptr;
    bool resident_pending = false;
    int state = kCreated;
    bool resident_set = false;
    bool primed = false;
    int k = 0;
    std::vector<const uint8_t*> host;
    std::vector<const uint8_t*> host_dev;
    std::vector<std::pair<void*, size_t>> reg_ranges;
    bool reg_read_only = false;
    bool pageable = false;
    uint8_t* hstage[2] = {nullptr, nullptr};   // pinned host staging slots (pageable mode)
    unsigned long long pack_seq = 0;            // pageable stagings so far (host slot = seq % 2)
    std::unique_ptr<HostPacker> packer;
    std::vector<uint8_t*> resident;
    unsigned long long exec_counter = 0;
    int slot_block[2] = {-1, -1};
    dlo_stats st{};
    std::vector<int> log_kind, log_block, log_slot;
    size_t log_total = 0;
    int timing = 0;
    std::vector<TimedExec> timed_pending;
    std::vector<TimedKernel> kernels_pending;
    std::vector<cudaEvent_t> ev_pool;
    std::string err;

    // Whole-forward CUDA graphs (dlo_set_graphs): executable graphs keyed by
    // the forward's arguments and the parity of exec_counter at its start
    // (the slot that holds the first streamed block), each with the host-side
    // effects of that forward (counters, log entries, slot contents) that are
    // replayed on each launch.  Up to kGraphs, least recently used replaced.
    static constexpr int kGraphs = 4;
    struct GraphRec {
        cudaGraphExec_t exec = nullptr;
        int par = 0;
        int timing = 0;                 // timing level the graph was captured at (0 or 3)
        std::vector<TimedKernel> tk;    // level 3: the kernel event pairs inside the graph
        bool tk_pending = false;        // a launch's pairs not read yet
        unsigned long long last_use = 0;
        const void* x_in = nullptr;
        std::vector<const void*> conds;
        const void* ctx = nullptr;
        void* x_out = nullptr;
        int B = 0, N = 0, L = 0;
        unsigned long long d_stagings = 0, d_staged_bytes = 0, d_streamed = 0, d_launches = 0,
                           d_h2d = 0, d_exec = 0;
        std::vector<int> lk, lb, ls;
        int slot_block_after[2] = {-1, -1};
    };
    int graphs = 0;
    bool capturing = false;
    bool cap_copy[2] = {false, false};    // copy_done[i] recorded inside the capture
    bool cap_comp[2] = {false, false};    // compute_done[i] recorded inside the capture
    GraphRec gr[kGraphs];
    unsigned long long graph_uses = 0;
    cudaEvent_t g_ev[2] = {nullptr, nullptr};
    void drop_graphs() {
        bool events = false;
        for (GraphRec& g : gr) events |= !g.tk.empty();
        // a graph's event pairs may still be recorded by a launch in flight
        if (events) cudaStreamSynchronize(cs);
        for (GraphRec& g : gr) {
            if (g.exec) cudaGraphExecDestroy(g.exec);
            for (TimedKernel& t : g.tk) {
                cudaEventDestroy(t.a);
                cudaEventDestroy(t.b);
            }
            g = GraphRec();
        }
    }

    dlo_status fail(dlo_status s, const char* fmt, ...) {
        char buf[512];
        va_list ap;
        va_start(ap, fmt);
        vsnprintf(buf, sizeof(buf), fmt, ap);
        va_end(ap);
        err = buf;
        return s;
    }
    dlo_status cuda_fail(cudaError_t e, const char* what) {
        return fail(DLO_ECUDA, "%s: %s (%d)", what, cudaGetErrorString(e), static_cast<int>(e));
    }
    void log(int kind, int block, int slot_) {
        ++log_total;
        if (log_kind.size() < 65536) {
            log_kind.push_back(kind);
            log_block.push_back(block);
            log_slot.push_back(slot_);
        }
    }
    bool any_video = false;
    int* err_word() { return reinterpret_cast<int*>(wsp + ws.err); }
    const Container& cont(int blk) const { return conts[cont_of[blk]]; }
    size_t bytes_of(int blk) const { return conts[cont_of[blk]].block_bytes; }
    // Launch through f(); with timing level 2 or 3 bracket it with events on
    // `s` and remember its class and algorithmic work.  Inside a graph
    // capture (level 3) the records are external event-record nodes, so the
    // events are recorded each time the graph runs.
    template <class Fn>
    cudaError_t timed(int cls, double flops, double bytes, cudaStream_t s, Fn f) {
        if (timing < 2) return f();
        TimedKernel t{cls, get_event(), get_event(), flops, bytes};
        const unsigned fl = capturing ? cudaEventRecordExternal : cudaEventRecordDefault;
        cudaError_t e = cudaEventRecordWithFlags(t.a, s, fl);
        if (e == cudaSuccess) e = f();
        if (e == cudaSuccess) e = cudaEventRecordWithFlags(t.b, s, fl);
        kernels_pending.push_back(t);
        return e;
    }
    cudaEvent_t get_event() {
        if (!ev_pool.empty()) {
            cudaEvent_t e = ev_pool.back();
            ev_pool.pop_back();
            return e;
        }
        cudaEvent_t e = nullptr;
        cudaEventCreate(&e);
        return e;
    }
};

namespace {

size_t off_of(const std::vector<Entry>& L, const char* n) {
    const int i = find_entry(L, n);
    return i < 0 ? 0 : L[i].offset;
}

void fill_offsets(Container* k) {
    const auto& L = k->L;
    Offsets& o = k->off;
    if (k->d.block_kind == DLO_BLOCK_DIT) {
        o.ada_w = off_of(L, "adaLN.weight");
        o.ada_b = off_of(L, "adaLN.bias");
        o.qkv_w = off_of(L, "attn.qkv.weight");
        o.qkv_b = off_of(L, "attn.qkv.bias");
        o.proj_w = off_of(L, "attn.proj.weight");
        o.proj_b = off_of(L, "attn.proj.bias");
        o.fc1_w = off_of(L, "mlp.fc1.weight");
        o.fc1_b = off_of(L, "mlp.fc1.bias");
        o.fc2_w = off_of(L, "mlp.fc2.weight");
        o.fc2_b = off_of(L, "mlp.fc2.bias");
        o.has_scales = false;
    } else {
        o.mod = off_of(L, "modulation");
        o.sq_w = off_of(L, "self_attn.q.weight");
        o.sq_b = off_of(L, "self_attn.q.bias");
        o.so_w = off_of(L, "self_attn.o.weight");
        o.so_b = off_of(L, "self_attn.o.bias");
        o.snq = off_of(L, "self_attn.norm_q.weight");
        o.snk = off_of(L, "self_attn.norm_k.weight");
        o.ncw = off_of(L, "norm_cross.weight");
        o.ncb = off_of(L, "norm_cross.bias");
        o.cq_w = off_of(L, "cross_attn.q.weight");
        o.cq_b = off_of(L, "cross_attn.q.bias");
        o.ck_w = off_of(L, "cross_attn.k.weight");
        o.ck_b = off_of(L, "cross_attn.k.bias");
        o.co_w = off_of(L, "cross_attn.o.weight");
        o.co_b = off_of(L, "cross_attn.o.bias");
        o.cnq = off_of(L, "cross_attn.norm_q.weight");
        o.cnk = off_of(L, "cross_attn.norm_k.weight");
        o.fc1_w = off_of(L, "ffn.fc1.weight");
        o.fc1_b = off_of(L, "ffn.fc1.bias");
        o.fc2_w = off_of(L, "ffn.fc2.weight");
        o.fc2_b = off_of(L, "ffn.fc2.bias");
        o.has_scales = find_entry(L, "linear_scales") >= 0;
        o.scales = off_of(L, "linear_scales");
    }
}

// Poll a stream until idle or the limit runs out: yielding between queries
// for the first 20 ms (a step's result is noticed within microseconds), then
// sleeping 50 us between them.
bool stream_wait(cudaStream_t s, int timeout_ms, cudaError_t* e) {
    const auto t0 = std::chrono::steady_clock::now();
    for (;;) {
        cudaError_t q = cudaStreamQuery(s);
        if (q == cudaSuccess) return true;
        if (q != cudaErrorNotReady) {
            *e = q;
            return false;
        }
        const auto us = std::chrono::duration_cast<std::chrono::microseconds>(
                            std::chrono::steady_clock::now() - t0).count();
        if (us > static_cast<long long>(timeout_ms) * 1000) {
            *e = cudaErrorNotReady;
            return false;
        }
        if (us < 20000)
            std::this_thread::yield();
        else
            std::this_thread::sleep_for(std::chrono::microseconds(50));
    }
}

// Copy host block `blk` into slot `s` on the copy stream.
dlo_status stage(dlo_ctx* c, int blk, int s) {
    cudaError_t e;
    const size_t bytes = c->bytes_of(blk);
    if (c->d.staging == DLO_STAGE_GATHER) {
        e = c->timed(DLO_K_GATHER, 0.0, 2.0 * bytes, c->xs, [&] {
            return launch_gather(c->slot[s], c->host_dev[blk], bytes, c->xs, &c->st.kernel_launches);
        });
    } else if (c->pageable) {
        // the packer thread packs the block into the next pinned host slot as
        // soon as that slot's previous copy has finished; the copy stream
        // waits for the pack, copies the slot and reports the copy
        const unsigned long long n = c->pack_seq;
        const int h = static_cast<int>(n & 1);
        PackTicket* w = new PackTicket{c->packer.get(), n};
        e = cudaLaunchHostFunc(c->xs, wait_packed_fn, w);
        if (e != cudaSuccess) {
            delete w;
        } else {
            c->packer->submit(n, c->hstage[h], c->host[blk], bytes);
            ++c->pack_seq;
            e = cudaMemcpyAsync(c->slot[s], c->hstage[h], bytes, cudaMemcpyHostToDevice, c->xs);
            ++c->st.h2d_copies;
            if (e == cudaSuccess) {
                PackTicket* d = new PackTicket{c->packer.get(), n};
                e = cudaLaunchHostFunc(c->xs, copied_fn, d);
                if (e != cudaSuccess) delete d;
            }
            // a copy that was not enqueued never reports: later packs into
            // this slot would wait for it, so the context takes no more work
            if (e != cudaSuccess) c->state = kBroken;
        }
    } else if (c->d.staging == DLO_STAGE_PER_TENSOR) {
        e = cudaSuccess;
        for (const Entry& t : c->cont(blk).L) {
            if (!t.bytes) continue;
            e = cudaMemcpyAsync(c->slot[s] + t.offset, c->host[blk] + t.offset, t.bytes,
                                cudaMemcpyHostToDevice, c->xs);
            if (e != cudaSuccess) break;
            ++c->st.h2d_copies;
        }
    } else {
        e = cudaMemcpyAsync(c->slot[s], c->host[blk], bytes, cudaMemcpyHostToDevice, c->xs);
        ++c->st.h2d_copies;
    }
    if (e != cudaSuccess) return c->cuda_fail(e, "slot staging");
    c->slot_block[s] = blk;
    ++c->st.stagings;
    c->st.staged_bytes += bytes;
    c->log(0, blk, s);
    return DLO_OK;
}

dlo_status prime(dlo_ctx* c) {
    if (c->primed) return DLO_OK;
    if (c->k < c->d.n_blocks) {
        dlo_status r = stage(c, c->k, 0);
        if (r != DLO_OK) return r;
        cudaError_t e = cudaEventRecord(c->copy_done[0], c->xs);
        if (e != cudaSuccess) return c->cuda_fail(e, "event record");
    }
    c->primed = true;
    return DLO_OK;
}

#define LCHECK(expr, what)                                   \
    do {                                                     \
        cudaError_t e_ = (expr);                             \
        if (e_ != cudaSuccess) return c->cuda_fail(e_, what); \
    } while (0)

// One block from weights at `W` (a slot or a resident buffer).
dlo_status run_block(dlo_ctx* c, const uint8_t* W, int B, int N, int L, const void* cond,
                     const void* ctx_tokens, int block, void* x_out) {
    const Container& K = c->cont(block);
    const dlo_desc& d = K.d;
    if (d.block_kind == DLO_BLOCK_BYTES) {
        unsigned long long* sums = static_cast<unsigned long long*>(x_out) + block;
        LCHECK(c->timed(DLO_K_CONVERT, 0.0, static_cast<double>(K.block_bytes), c->cs, [&] {
                   return launch_checksum(W, K.block_bytes, sums, c->cs, &c->st.kernel_launches);
               }),
               "checksum");
        return DLO_OK;
    }
    const Offsets& o = K.off;
    const int D = d.hidden, F = d.ffn, H = d.heads, hd = d.head_dim;
    const int BN = B * N;
    uint8_t* w = c->wsp;
    float* x = reinterpret_cast<float*>(w + c->ws.x);
    void* h = w + c->ws.h;
    void* big = w + c->ws.big;
    void* a = w + c->ws.a;
    float* m = reinterpret_cast<float*>(w + c->ws.mod);
    unsigned long long* nl = &c->st.kernel_launches;
    cudaStream_t s = c->cs;
    const int D6 = 6 * D;
    const bool e4m3 = e4m3_weights(d.wdtype);
    const bool w8a8 = d.wdtype == DLO_W_E4M3_A8;
    const int wsize = e4m3 ? 1 : 2;
    auto gemm = [&](const void* A, size_t woff, size_t boff, int M, int Nn, int K, int epi,
                    void* out, int ldo, const float* gate, int rpb, int scale_idx, int seg) {
        GemmParams p;
        p.A = A;
        if (w8a8) {
            // quantise this linear's input (dynamic per-tensor scale), then
            // multiply E4M3 by E4M3
            uint8_t* qa = w + c->ws.qa;
            float* part = reinterpret_cast<float*>(w + c->ws.qs);
            float* sx = part + kQuantScratch;
            cudaError_t e = c->timed(DLO_K_QUANT, 0.0, 5.0 * M * K, s, [&] {
                return launch_quantize_e4m3(A, M, K, K, qa, sx, part, s, nl);
            });
            if (e != cudaSuccess) return e;
            p.A = qa;
            p.a_dtype = DLO_DT_E4M3;
            p.a_scale = sx;
        }
        p.W = W + woff;
        p.w_dtype = e4m3 ? DLO_DT_E4M3 : DLO_DT_BF16;
        p.w_ready = true;   // weights live in a slot or resident buffer, never a kernel's output
        p.scales = o.has_scales ? reinterpret_cast<const float*>(W + o.scales) + scale_idx : nullptr;
        p.scale_seg = seg;
        p.bias = W + boff;
        p.M = M;
        p.N = Nn;
        p.K = K;
        p.epi = epi;
        p.out = out;
        p.ldo = ldo;
        p.gate = gate;
        p.gate_ld = D6;
        p.rows_per_batch = rpb;
        p.err = c->err_word();
        const double flops = 2.0 * M * Nn * K;
        const size_t nk = static_cast<size_t>(Nn) * K;
        auto bytes_of = [&](double w_bytes) {
            return 1.0 * M * K * (w8a8 ? 1 : 2) + w_bytes + 1.0 * M * Nn * (epi == DLO_EPI_RESIDUAL ? 8 : 2);
        };
        const int cls = w8a8 ? DLO_K_GEMM_FP8 : e4m3 ? DLO_K_GEMM_E4M3 : DLO_K_GEMM_BF16;
        // W8A16 at many rows: the GEMM kernel first widens this linear's codes
        // to bf16 in a workspace buffer (every CTA a share, then a grid
        // barrier) and then multiplies in bf16 on CTA pairs, which outpaces
        // widening each tile inside every CTA's mainloop; the per-tensor scale
        // stays in the epilogue, so the products are the same.  Where that
        // kernel form is unavailable, a separate widening kernel runs first.
        const bool widen = e4m3 && !w8a8 && M >= widen_rows() && nk * 2 <= c->ws.wide_bytes &&
                           (reinterpret_cast<uintptr_t>(p.W) & 15) == 0;
        if (widen) {
            void* wide = w + c->ws.wide;
            GemmParams q = p;
            q.w_codes = p.W;
            q.W = wide;
            q.w_dtype = DLO_DT_BF16;
            q.w_sync = reinterpret_cast<unsigned*>(w + c->ws.gsync);
            q.w_ready = false;
            cudaError_t e = c->timed(cls, flops, bytes_of(1.0 * nk), s, [&] { return launch_gemm(q, s, nl); });
            if (e != cudaErrorNotSupported) return e;
            e = c->timed(DLO_K_CONVERT, 0.0, 3.0 * nk, s, [&] { return launch_widen_e4m3(p.W, nk, wide, s, nl); });
            if (e != cudaSuccess) return e;
            p.W = wide;
            p.w_dtype = DLO_DT_BF16;
            p.w_ready = false;   // the widening kernel just wrote it
        }
        return c->timed(cls, flops, bytes_of(1.0 * nk * (widen ? 2 : wsize)), s,
                        [&] { return launch_gemm(p, s, nl); });
    };
    auto attn = [&](const void* q, const void* k, const void* v, void* out, int nq, int nk, int ldq, int ldk,
                    int ldv) {
        const double flops = 4.0 * B * H * nq * static_cast<double>(nk) * hd;
        const double bytes = 2.0 * B * (2.0 * nq + 2.0 * nk) * D;
        return c->timed(DLO_K_ATTENTION, flops, bytes, s, [&] {
            return launch_attention(q, k, v, out, B, H, hd, nq, nk, ldq, ldk, ldv, D, c->err_word(), s, nl);
        });
    };
    auto ln = [&](const float* shift, const float* scale, const void* lw, const void* lb) {
        return c->timed(DLO_K_LAYERNORM, 0.0, 6.0 * BN * D, s, [&] {
            return launch_layernorm(x, BN, D, N, shift, scale, D6, lw, lb, d.eps, h, s, nl);
        });
    };
    char* bigc = static_cast<char*>(big);
    if (d.block_kind == DLO_BLOCK_DIT) {
        LCHECK(c->timed(DLO_K_MODULATION, 2.0 * B * D6 * d.cond_dim, 2.0 * D6 * d.cond_dim, s,
                        [&] { return launch_adaln(cond, B, d.cond_dim, W + o.ada_w, W + o.ada_b, D6, m, s, nl, true); }),
               "adaLN");
        LCHECK(ln(m, m + D, nullptr, nullptr), "LN1");
        LCHECK(gemm(h, o.qkv_w, o.qkv_b, BN, 3 * D, D, DLO_EPI_BIAS, big, 3 * D, nullptr, N, 0, 3 * D), "qkv");
        LCHECK(attn(big, bigc + 2 * D, bigc + 4 * D, a, N, N, 3 * D, 3 * D, 3 * D), "attention");
        LCHECK(gemm(a, o.proj_w, o.proj_b, BN, D, D, DLO_EPI_RESIDUAL, x, D, m + 2 * D, N, 0, D), "proj");
        LCHECK(ln(m + 3 * D, m + 4 * D, nullptr, nullptr), "LN2");
        LCHECK(gemm(h, o.fc1_w, o.fc1_b, BN, F, D, DLO_EPI_GELU, big, F, nullptr, N, 0, F), "fc1");
        LCHECK(gemm(big, o.fc2_w, o.fc2_b, BN, D, F, DLO_EPI_RESIDUAL, x, D, m + 5 * D, N, 0, D), "fc2");
        return DLO_OK;
    }
    void* q2 = w + c->ws.q2;
    void* kv2 = w + c->ws.kv2;
    char* kv2c = static_cast<char*>(kv2);
    const int Dt = d.text_dim;
    LCHECK(c->timed(DLO_K_MODULATION, 0.0, 10.0 * B * D6, s,
                    [&] { return launch_mod_add(static_cast<const float*>(cond), W + o.mod, B, D6, m, s, nl); }),
           "modulation");
    LCHECK(ln(m, m + D, nullptr, nullptr), "LN1");
    LCHECK(gemm(h, o.sq_w, o.sq_b, BN, 3 * D, D, DLO_EPI_BIAS, big, 3 * D, nullptr, N, 0, D), "self qkv");
    LCHECK(c->timed(DLO_K_RMSNORM, 0.0, 8.0 * BN * D, s,
                    [&] { return launch_rmsnorm2(big, BN, D, 3 * D, 0, W + o.snq, D, W + o.snk, d.eps, s, nl); }),
           "self q/k norm");
    LCHECK(attn(big, bigc + 2 * D, bigc + 4 * D, a, N, N, 3 * D, 3 * D, 3 * D), "self attention");
    LCHECK(gemm(a, o.so_w, o.so_b, BN, D, D, DLO_EPI_RESIDUAL, x, D, m + 2 * D, N, 3, D), "self o");
    LCHECK(ln(nullptr, nullptr, W + o.ncw, W + o.ncb), "LN cross");
    LCHECK(gemm(h, o.cq_w, o.cq_b, BN, D, D, DLO_EPI_BIAS, q2, D, nullptr, N, 4, D), "cross q");
    LCHECK(gemm(ctx_tokens, o.ck_w, o.ck_b, B * L, 2 * D, Dt, DLO_EPI_BIAS, kv2, 2 * D, nullptr, L, 5, D),
           "cross kv");
    LCHECK(c->timed(DLO_K_RMSNORM, 0.0, 4.0 * BN * D, s,
                    [&] { return launch_rmsnorm(q2, BN, D, D, 0, W + o.cnq, d.eps, s, nl); }),
           "cross q norm");
    LCHECK(c->timed(DLO_K_RMSNORM, 0.0, 4.0 * B * L * D, s,
                    [&] { return launch_rmsnorm(kv2, B * L, D, 2 * D, 0, W + o.cnk, d.eps, s, nl); }),
           "cross k norm");
    LCHECK(attn(q2, kv2, kv2c + 2 * D, a, N, L, D, 2 * D, 2 * D), "cross attention");
    LCHECK(gemm(a, o.co_w, o.co_b, BN, D, D, DLO_EPI_RESIDUAL, x, D, nullptr, N, 7, D), "cross o");
    LCHECK(ln(m + 3 * D, m + 4 * D, nullptr, nullptr), "LN2");
    LCHECK(gemm(h, o.fc1_w, o.fc1_b, BN, F, D, DLO_EPI_GELU, big, F, nullptr, N, 8, F), "fc1");
    LCHECK(gemm(big, o.fc2_w, o.fc2_b, BN, D, F, DLO_EPI_RESIDUAL, x, D, m + 5 * D, N, 9, D), "fc2");
    return DLO_OK;
}

// The kernel event pairs of the last launch of each graph captured at timing
// level 3, once that launch has run (wait: block until it has).
void collect_graph_timing(dlo_ctx* c, bool wait) {
    for (dlo_ctx::GraphRec& g : c->gr) {
        if (!g.tk_pending) continue;
        if (wait) cudaEventSynchronize(g.tk.back().b);
        float probe = 0;
        if (cudaEventElapsedTime(&probe, g.tk.back().a, g.tk.back().b) != cudaSuccess) {
            cudaGetLastError();
            continue;   // still running
        }
        for (TimedKernel& t : g.tk) {
            float ms = 0;
            if (cudaEventElapsedTime(&ms, t.a, t.b) != cudaSuccess) {
                cudaGetLastError();
                continue;
            }
            c->st.kclass_ms[t.cls] += ms;
            c->st.kclass_flops[t.cls] += t.flops;
            c->st.kclass_bytes[t.cls] += t.bytes;
            ++c->st.kclass_launches[t.cls];
        }
        g.tk_pending = false;
    }
}

void collect_timing(dlo_ctx* c) {
    collect_graph_timing(c, false);
    std::vector<TimedExec> keep;
    for (auto& t : c->timed_pending) {
        float cp = 0, cm = 0, wt = 0;
        if (cudaEventElapsedTime(&cp, t.copy0, t.copy1) != cudaSuccess ||
            cudaEventElapsedTime(&cm, t.comp0, t.comp1) != cudaSuccess ||
            cudaEventElapsedTime(&wt, t.wait0, t.comp0) != cudaSuccess) {
            cudaGetLastError();
            keep.push_back(t);
            continue;
        }
        c->st.copy_ms += cp;
        c->st.compute_ms += cm;
        c->st.exposed_wait_ms += wt;
        ++c->st.timed_execs;
        for (cudaEvent_t e : {t.copy0, t.copy1, t.wait0, t.comp0, t.comp1}) c->ev_pool.push_back(e);
    }
    c->timed_pending.swap(keep);
    std::vector<TimedKernel> kk;
    for (auto& t : c->kernels_pending) {
        float ms = 0;
        if (cudaEventElapsedTime(&ms, t.a, t.b) != cudaSuccess) {
            cudaGetLastError();
            kk.push_back(t);
            continue;
        }
        c->st.kclass_ms[t.cls] += ms;
        c->st.kclass_flops[t.cls] += t.flops;
        c->st.kclass_bytes[t.cls] += t.bytes;
        ++c->st.kclass_launches[t.cls];
        c->ev_pool.push_back(t.a);
        c->ev_pool.push_back(t.b);
    }
    c->kernels_pending.swap(kk);
}

dlo_status check_device_error(dlo_ctx* c) {
    int v = 0;
    cudaError_t e = cudaMemcpy(&v, c->err_word(), sizeof(int), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return c->cuda_fail(e, "reading the kernels' error word");
    c->st.device_error = v;
    if (v) {
        cudaMemset(c->err_word(), 0, sizeof(int));
        return c->fail(DLO_ETIMEDOUT, "a kernel's bounded wait ran out (error word %d)", v);
    }
    return DLO_OK;
}

}  // namespace

// ===================================================================== C ABI

extern "C" const char* dlo_last_error(const dlo_ctx* ctx) {
    if (!ctx) return g_create_error.c_str();
    return ctx->err.c_str();
}

extern "C" void dlo_debug_fail_register(int nth) { g_fail_register_nth.store(nth > 0 ? nth : 0); }

namespace {

dlo_status create_stack(const dlo_desc* descs, int n_cont, int device, void* slot0, void* slot1,
                        size_t slot_bytes, void* workspace, size_t ws_bytes, void* compute_stream,
                        void* copy_stream, dlo_ctx** out) {
    if (out) *out = nullptr;
    std::string msg;
    dlo_desc whole{};
    dlo_status st = validate_stack(descs, n_cont, &whole, &msg);
    auto cfail = [&](dlo_status s, const std::string& m) {
        g_create_error = m;
        return s;
    };
    if (!out) return cfail(DLO_EINVAL, "out is NULL");
    if (st != DLO_OK) return cfail(st, msg);
    std::vector<Container> conts(n_cont);
    std::vector<int> cont_of;
    size_t bb = 0;
    for (int i = 0; i < n_cont; ++i) {
        conts[i].d = descs[i];
        conts[i].block_bytes = build_layout(descs[i], &conts[i].L);
        conts[i].first = static_cast<int>(cont_of.size());
        fill_offsets(&conts[i]);
        cont_of.insert(cont_of.end(), descs[i].n_blocks, i);
        bb = std::max(bb, conts[i].block_bytes);
    }
    const Workspace ws = plan_workspace_stack(descs, n_cont);
    if (!slot0 || !slot1 || slot0 == slot1) return cfail(DLO_EINVAL, "two distinct slots are required");
    if (!aligned(slot0, 256) || !aligned(slot1, 256) || !aligned(workspace, 256))
        return cfail(DLO_EINVAL, "slots and workspace must be 256-byte aligned");
    if (slot_bytes < bb) return cfail(DLO_ENOMEM, "slot_bytes < bytes of the largest block");
    {
        const uintptr_t a0 = reinterpret_cast<uintptr_t>(slot0), a1 = reinterpret_cast<uintptr_t>(slot1);
        if ((a0 < a1 && a0 + slot_bytes > a1) || (a1 < a0 && a1 + slot_bytes > a0))
            return cfail(DLO_EINVAL, "slots overlap");
    }
    if (!workspace || ws_bytes < ws.total) return cfail(DLO_ENOMEM, "workspace too small");
    if (!compute_stream || !copy_stream || compute_stream == copy_stream)
        return cfail(DLO_EINVAL, "distinct non-NULL compute and copy streams are required");
    int ndev = 0;
    cudaError_t e = cudaGetDeviceCount(&ndev);
    if (e != cudaSuccess) return cfail(DLO_ECUDA, std::string("cudaGetDeviceCount: ") + cudaGetErrorString(e));
    if (device < 0 || device >= ndev) return cfail(DLO_EINVAL, "bad device ordinal");
    e = cudaSetDevice(device);
    if (e != cudaSuccess) return cfail(DLO_ECUDA, std::string("cudaSetDevice: ") + cudaGetErrorString(e));

    std::unique_ptr<dlo_ctx> c(new dlo_ctx());
    c->d = whole;
    c->device = device;
    c->conts = std::move(conts);
    c->cont_of = std::move(cont_of);
    for (const Container& k : c->conts) c->any_video |= k.d.block_kind == DLO_BLOCK_VIDEO;
    c->block_bytes = bb;
    c->ws = ws;
    c->slot[0] = static_cast<uint8_t*>(slot0);
    c->slot[1] = static_cast<uint8_t*>(slot1);
    c->slot_bytes = slot_bytes;
    c->wsp = static_cast<uint8_t*>(workspace);
    c->cs = static_cast<cudaStream_t>(compute_stream);
    c->xs = static_cast<cudaStream_t>(copy_stream);
    auto evfail = [&](cudaError_t err) {
        for (int i = 0; i < 2; ++i) {
            if (c->copy_done[i]) cudaEventDestroy(c->copy_done[i]);
            if (c->compute_done[i]) cudaEventDestroy(c->compute_done[i]);
        }
        if (c->resident_ev) cudaEventDestroy(c->resident_ev);
        return cfail(DLO_ECUDA, std::string("event create: ") + cudaGetErrorString(err));
    };
    for (int i = 0; i < 2; ++i) {
        if ((e = cudaEventCreateWithFlags(&c->copy_done[i], cudaEventDisableTiming)) != cudaSuccess) return evfail(e);
        if ((e = cudaEventCreateWithFlags(&c->compute_done[i], cudaEventDisableTiming)) != cudaSuccess)
            return evfail(e);
    }
    if ((e = cudaEventCreateWithFlags(&c->resident_ev, cudaEventDisableTiming)) != cudaSuccess) return evfail(e);
    e = cudaMemsetAsync(c->err_word(), 0, 64 * sizeof(int), c->cs);
    if (e != cudaSuccess) return evfail(e);
    gemm_num_sms();
    c->st.slot_block[0] = c->st.slot_block[1] = -1;
    *out = c.release();
    return DLO_OK;
}

}  // namespace

extern "C" dlo_status dlo_create(const dlo_desc* desc, int device, void* slot0, void* slot1,
                                 size_t slot_bytes, void* workspace, size_t ws_bytes,
                                 void* compute_stream, void* copy_stream, dlo_ctx** out) {
    return create_stack(desc, 1, device, slot0, slot1, slot_bytes, workspace, ws_bytes, compute_stream,
                        copy_stream, out);
}

extern "C" dlo_status dlo_create_multi(const dlo_desc* descs, int n_containers, int device, void* slot0,
                                       void* slot1, size_t slot_bytes, void* workspace, size_t ws_bytes,
                                       void* compute_stream, void* copy_stream, dlo_ctx** out) {
    return create_stack(descs, n_containers, device, slot0, slot1, slot_bytes, workspace, ws_bytes,
                        compute_stream, copy_stream, out);
}

extern "C" dlo_status dlo_register_host_blocks(dlo_ctx* c, int n, const void* const* host_blocks,
                                               size_t block_bytes, unsigned flags) {
    if (!c) return DLO_EINVAL;
    if (c->state != kCreated) return c->fail(DLO_ESTATE, "host blocks are already attached");
    if (n != c->d.n_blocks) return c->fail(DLO_EINVAL, "n (%d) != n_blocks (%d)", n, c->d.n_blocks);
    if (!host_blocks) return c->fail(DLO_EINVAL, "host_blocks is NULL");
    if (block_bytes != 0 && (c->conts.size() != 1 || block_bytes != c->block_bytes))
        return c->fail(DLO_EINVAL, "block_bytes %zu != layout bytes %zu (pass 0 to use each block's own size)",
                       block_bytes, c->block_bytes);
    const bool pinned = flags == DLO_HOST_PINNED, reg = flags == DLO_HOST_REGISTER;
    const bool pageable = flags == DLO_HOST_PAGEABLE;
    if (!pinned && !reg && !pageable)
        return c->fail(DLO_EINVAL, "flags must be one of DLO_HOST_PINNED, DLO_HOST_REGISTER, DLO_HOST_PAGEABLE");
    if (pageable && c->d.staging != DLO_STAGE_MEMCPY)
        return c->fail(DLO_EINVAL, "DLO_HOST_PAGEABLE needs DLO_STAGE_MEMCPY");
    for (int i = 0; i < n; ++i) {
        if (!host_blocks[i]) return c->fail(DLO_EINVAL, "host block %d is NULL", i);
        if (!aligned(host_blocks[i], 16)) return c->fail(DLO_EINVAL, "host block %d is not 16-byte aligned", i);
    }
    cudaSetDevice(c->device);
    if (pageable) {
        // two bounded pinned host staging slots; nothing else is page-locked
        for (int i = 0; i < 2; ++i) {
            cudaError_t e = cudaHostAlloc(reinterpret_cast<void**>(&c->hstage[i]), c->block_bytes,
                                          cudaHostAllocDefault);
            if (e != cudaSuccess) {
                cudaGetLastError();
                for (int k = 0; k < i; ++k) cudaFreeHost(c->hstage[k]);
                c->hstage[0] = c->hstage[1] = nullptr;
                return c->fail(DLO_ENOMEM, "pinned host staging slots: %s", cudaGetErrorString(e));
            }
        }
        c->packer.reset(new HostPacker(pack_threads()));
        c->pageable = true;
        c->host.assign(reinterpret_cast<const uint8_t* const*>(host_blocks),
                       reinterpret_cast<const uint8_t* const*>(host_blocks) + n);
        c->host_dev.assign(n, nullptr);
        c->state = kRegistered;
        return DLO_OK;
    }
    std::vector<std::pair<void*, size_t>> done;
    bool ro = false;
    if (reg) {
        // page-align the block ranges and merge overlapping or adjacent ones
        const size_t page = 4096;
        std::vector<std::pair<uintptr_t, uintptr_t>> r;
        for (int i = 0; i < n; ++i) {
            const uintptr_t a = reinterpret_cast<uintptr_t>(host_blocks[i]);
            r.push_back({a / page * page, (a + c->bytes_of(i) + page - 1) / page * page});
        }
        std::sort(r.begin(), r.end());
        std::vector<std::pair<uintptr_t, uintptr_t>> merged;
        for (auto& x : r) {
            if (!merged.empty() && x.first <= merged.back().second)
                merged.back().second = std::max(merged.back().second, x.second);
            else
                merged.push_back(x);
        }
        unsigned long long total = 0;
        for (auto& x : merged) total += x.second - x.first;
        if (c->d.register_budget_bytes && total > c->d.register_budget_bytes)
            return c->fail(DLO_EREGISTER, "registration needs %llu bytes, budget is %llu (nothing registered)",
                           total, c->d.register_budget_bytes);
        int ro_ok = 0;
        cudaDeviceGetAttribute(&ro_ok, cudaDevAttrHostRegisterReadOnlySupported, c->device);
        ro = ro_ok != 0;
        const unsigned rflags = cudaHostRegisterPortable | cudaHostRegisterMapped | (ro ? cudaHostRegisterReadOnly : 0u);
        for (auto& x : merged) {
            void* p = reinterpret_cast<void*>(x.first);
            const size_t len = x.second - x.first;
            cudaError_t e;
            int nth = g_fail_register_nth.load();
            if (nth > 0 && g_fail_register_nth.fetch_sub(1) == 1) {
                e = cudaErrorHostMemoryAlreadyRegistered;   // injected failure; no call made
            } else {
                e = cudaHostRegister(p, len, rflags);
            }
            if (e != cudaSuccess) {
                cudaGetLastError();
                std::string why = cudaGetErrorString(e);
                bool rollback_ok = true;
                for (auto& u : done) {
                    if (cudaHostUnregister(u.first) != cudaSuccess) {
                        cudaGetLastError();
                        rollback_ok = false;
                        c->reg_ranges.push_back(u);   // still registered: destroy retries
                    }
                }
                if (!rollback_ok) {
                    c->state = kBroken;
                    return c->fail(DLO_EREGISTER,
                                   "cudaHostRegister failed (%s) and the rollback failed; the context "
                                   "is unusable, destroy it",
                                   why.c_str());
                }
                return c->fail(DLO_EREGISTER, "cudaHostRegister of %zu bytes failed (%s); %zu ranges rolled back",
                               len, why.c_str(), done.size());
            }
            done.push_back({p, len});
        }
    }
    // every block must read as page-locked host memory; record device addresses
    std::vector<const uint8_t*> hd(n);
    for (int i = 0; i < n; ++i) {
        cudaPointerAttributes at{};
        cudaError_t e = cudaPointerGetAttributes(&at, host_blocks[i]);
        const uint8_t* last = static_cast<const uint8_t*>(host_blocks[i]) + c->bytes_of(i) - 1;
        cudaPointerAttributes at2{};
        cudaError_t e2 = cudaPointerGetAttributes(&at2, last);
        if (e != cudaSuccess || e2 != cudaSuccess || at.type != cudaMemoryTypeHost ||
            at2.type != cudaMemoryTypeHost) {
            cudaGetLastError();
            for (auto& u : done) cudaHostUnregister(u.first);
            cudaGetLastError();
            return c->fail(reg ? DLO_EREGISTER : DLO_EINVAL, "host block %d is not page-locked host memory", i);
        }
        hd[i] = static_cast<const uint8_t*>(at.devicePointer);
        if (c->d.staging == DLO_STAGE_GATHER && !hd[i]) {
            for (auto& u : done) cudaHostUnregister(u.first);
            cudaGetLastError();
            return c->fail(DLO_EINVAL, "host block %d is not mapped into the device address space", i);
        }
    }
    c->host.assign(reinterpret_cast<const uint8_t* const*>(host_blocks),
                   reinterpret_cast<const uint8_t* const*>(host_blocks) + n);
    c->host_dev = hd;
    c->reg_ranges.insert(c->reg_ranges.end(), done.begin(), done.end());
    c->reg_read_only = ro && !done.empty();
    c->state = kRegistered;
    return DLO_OK;
}

extern "C" dlo_status dlo_set_resident(dlo_ctx* c, int k, void* const* device_blocks) {
    if (!c) return DLO_EINVAL;
    if (c->state != kRegistered) return c->fail(DLO_ESTATE, "register host blocks first");
    if (c->resident_set || c->primed) return c->fail(DLO_ESTATE, "resident blocks must be set once, before the first forward");
    if (k < 0 || k > c->d.n_blocks) return c->fail(DLO_EINVAL, "k must be in [0, n_blocks]");
    if (k > 0 && !device_blocks) return c->fail(DLO_EINVAL, "device_blocks is NULL");
    for (int i = 0; i < k; ++i)
        if (!device_blocks[i] || !aligned(device_blocks[i], 256))
            return c->fail(DLO_EINVAL, "resident buffer %d is NULL or not 256-byte aligned", i);
    cudaSetDevice(c->device);
    for (int i = 0; i < k; ++i) {
        cudaError_t e = cudaMemcpyAsync(device_blocks[i], c->host[i], c->bytes_of(i), cudaMemcpyHostToDevice, c->xs);
        if (e != cudaSuccess) return c->cuda_fail(e, "resident copy");
    }
    if (k > 0) {
        cudaError_t e = cudaEventRecord(c->resident_ev, c->xs);
        if (e != cudaSuccess) return c->cuda_fail(e, "event record");
        c->resident_pending = true;
    }
    c->k = k;
    c->resident.assign(reinterpret_cast<uint8_t* const*>(device_blocks),
                       reinterpret_cast<uint8_t* const*>(device_blocks) + k);
    c->resident_set = true;
    c->st.resident = k;
    return prime(c);
}

namespace {

// One forward over every container's blocks in order; conds[i] conditions
// the blocks of container i.
dlo_status enqueue_forward(dlo_ctx* c, const void* x_in, const void* const* conds, const void* ctx_tokens,
                           int batch, int tokens, int text_tokens, void* x_out);
dlo_status forward_graph(dlo_ctx* c, const void* x_in, const void* const* conds, const void* ctx_tokens,
                         int batch, int tokens, int text_tokens, void* x_out);

dlo_status forward_stack(dlo_ctx* c, const void* x_in, const void* const* conds, const void* ctx_tokens,
                         int batch, int tokens, int text_tokens, void* x_out) {
    if (c->state != kRegistered) return c->fail(DLO_ESTATE, "register host blocks first");
    const dlo_desc& d = c->d;
    const bool bytes_kind = d.block_kind == DLO_BLOCK_BYTES;
    if (bytes_kind) {
        if (batch != 1 || tokens != 1) return c->fail(DLO_EINVAL, "bytes blocks take batch = tokens = 1");
        if (!x_out || !aligned(x_out, 8)) return c->fail(DLO_EINVAL, "x_out must be an 8-byte aligned uint64 array");
    } else {
    if (batch < 1 || batch > d.max_batch) return c->fail(DLO_EINVAL, "batch out of range");
    if (tokens < 1 || tokens > d.max_tokens) return c->fail(DLO_EINVAL, "tokens out of range");
    if (!x_in || !x_out) return c->fail(DLO_EINVAL, "NULL input/output");
    if (!aligned(x_in, 16) || !aligned(x_out, 16))
        return c->fail(DLO_EINVAL, "inputs/outputs must be 16-byte aligned");
    for (size_t i = 0; i < c->conts.size(); ++i)
        if (!conds[i] || !aligned(conds[i], 16))
            return c->fail(DLO_EINVAL, "conditioning of container %zu is NULL or not 16-byte aligned", i);
    if (c->any_video) {
        if (text_tokens < 1 || text_tokens > d.max_text_tokens) return c->fail(DLO_EINVAL, "text_tokens out of range");
        if (!ctx_tokens || !aligned(ctx_tokens, 16)) return c->fail(DLO_EINVAL, "ctx_tokens NULL or misaligned");
    }
    }
    cudaSetDevice(c->device);
    dlo_status r = prime(c);
    if (r != DLO_OK) return r;
    if (c->resident_pending) {
        LCHECK(cudaStreamWaitEvent(c->cs, c->resident_ev, 0), "wait resident");
        c->resident_pending = false;
    }
    // the first forward is enqueued directly: kernels' one-time set-up
    // (attributes, tensor-map encoders) runs outside any capture
    if (c->graphs && (c->timing == 0 || c->timing == 3) && !c->pageable && c->st.forwards > 0)
        r = forward_graph(c, x_in, conds, ctx_tokens, batch, tokens, text_tokens, x_out);
    else
        r = enqueue_forward(c, x_in, conds, ctx_tokens, batch, tokens, text_tokens, x_out);
    if (r == DLO_OK) ++c->st.forwards;
    return r;
}

// The stream work of one forward on the compute and copy streams.  While a
// graph is being captured, waits on events recorded before the capture are
// left out: the graph's launch is ordered after all earlier work of both
// streams (forward_graph).
dlo_status enqueue_forward(dlo_ctx* c, const void* x_in, const void* const* conds, const void* ctx_tokens,
                           int batch, int tokens, int text_tokens, void* x_out) {
    const dlo_desc& d = c->d;
    const bool bytes_kind = d.block_kind == DLO_BLOCK_BYTES;
    dlo_status r = DLO_OK;
    const int n = d.n_blocks, k = c->k;
    const size_t nx = bytes_kind ? 0 : static_cast<size_t>(batch) * tokens * d.hidden;
    float* x = reinterpret_cast<float*>(c->wsp + c->ws.x);
    if (bytes_kind) {
        LCHECK(cudaMemsetAsync(x_out, 0, static_cast<size_t>(n) * 8, c->cs), "clear checksums");
    } else {
        LCHECK(c->timed(DLO_K_CONVERT, 0.0, 6.0 * nx, c->cs,
                        [&] { return launch_bf16_to_f32(x_in, x, nx, c->cs, &c->st.kernel_launches); }),
               "input conversion");
    }
    for (int i = 0; i < k; ++i) {
        c->log(1, i, -1);
        r = run_block(c, c->resident[i], batch, tokens, text_tokens, conds[c->cont_of[i]], ctx_tokens, i, x_out);
        if (r != DLO_OK) return r;
    }
    for (int i = k; i < n; ++i) {
        const int s = static_cast<int>(c->exec_counter & 1), t = s ^ 1;
        const int nb = i < n - 1 ? i + 1 : k;
        TimedExec te{};
        const bool per_exec = c->timing == 1 || c->timing == 2;   // level 3 times kernels only
        if (per_exec) {
            te.copy0 = c->get_event();
            te.copy1 = c->get_event();
            te.wait0 = c->get_event();
            te.comp0 = c->get_event();
            te.comp1 = c->get_event();
        }
        // prefetch the next block into the other slot once its last reader is done
        if (!c->capturing || c->cap_comp[t])
            LCHECK(cudaStreamWaitEvent(c->xs, c->compute_done[t], 0), "copy waits compute");
        if (per_exec) LCHECK(cudaEventRecord(te.copy0, c->xs), "event");
        r = stage(c, nb, t);
        if (r != DLO_OK) return r;
        if (per_exec) LCHECK(cudaEventRecord(te.copy1, c->xs), "event");
        LCHECK(cudaEventRecord(c->copy_done[t], c->xs), "event record");
        c->cap_copy[t] = c->capturing;
        // compute block i from slot s once its copy landed
        if (per_exec) LCHECK(cudaEventRecord(te.wait0, c->cs), "event");
        if (!c->capturing || c->cap_copy[s])
            LCHECK(cudaStreamWaitEvent(c->cs, c->copy_done[s], 0), "compute waits copy");
        if (per_exec) LCHECK(cudaEventRecord(te.comp0, c->cs), "event");
        c->log(1, i, s);
        r = run_block(c, c->slot[s], batch, tokens, text_tokens, conds[c->cont_of[i]], ctx_tokens, i, x_out);
        if (r != DLO_OK) return r;
        if (per_exec) LCHECK(cudaEventRecord(te.comp1, c->cs), "event");
        LCHECK(cudaEventRecord(c->compute_done[s], c->cs), "event record");
        c->cap_comp[s] = c->capturing;
        if (per_exec) c->timed_pending.push_back(te);
        ++c->exec_counter;
        ++c->st.streamed_execs;
    }
    if (!bytes_kind) {
        LCHECK(c->timed(DLO_K_CONVERT, 0.0, 6.0 * nx, c->cs,
                        [&] { return launch_f32_to_bf16(x, x_out, nx, c->cs, &c->st.kernel_launches); }),
               "output conversion");
    }
    return DLO_OK;
}

// Host-side state a capture changes; restored when a capture fails (the
// captured work never ran).
struct HostSnap {
    dlo_stats st;
    size_t log_n, log_total;
    unsigned long long exec;
    int slot_block[2];
};

HostSnap snap(const dlo_ctx* c) {
    return HostSnap{c->st, c->log_kind.size(), c->log_total, c->exec_counter,
                    {c->slot_block[0], c->slot_block[1]}};
}

void restore(dlo_ctx* c, const HostSnap& h) {
    c->st = h.st;
    c->log_kind.resize(h.log_n);
    c->log_block.resize(h.log_n);
    c->log_slot.resize(h.log_n);
    c->log_total = h.log_total;
    c->exec_counter = h.exec;
    c->slot_block[0] = h.slot_block[0];
    c->slot_block[1] = h.slot_block[1];
}

// One forward as a CUDA graph: captured on first use for these arguments and
// this slot parity, then launched.  All earlier copy-stream work is joined
// into the compute stream before the launch; after it, the slot events are
// re-recorded on the compute stream so direct forwards and dlo_verify_slot
// see the graph's copies and computes as done.
dlo_status forward_graph(dlo_ctx* c, const void* x_in, const void* const* conds, const void* ctx_tokens,
                         int batch, int tokens, int text_tokens, void* x_out) {
    for (int i = 0; i < 2; ++i)
        if (!c->g_ev[i]) LCHECK(cudaEventCreateWithFlags(&c->g_ev[i], cudaEventDisableTiming), "event create");
    const size_t nc = c->conts.size();
    const int par = static_cast<int>(c->exec_counter & 1);
    dlo_ctx::GraphRec* found = nullptr;
    dlo_ctx::GraphRec* victim = nullptr;    // the first free entry, else the least recently used
    for (dlo_ctx::GraphRec& r : c->gr) {
        if (r.exec && r.par == par && r.timing == c->timing && r.x_in == x_in && r.ctx == ctx_tokens &&
            r.x_out == x_out &&
            r.B == batch && r.N == tokens && r.L == text_tokens &&
            std::equal(r.conds.begin(), r.conds.end(), conds, conds + nc)) {
            found = &r;
            break;
        }
        if (!r.exec) {
            if (!victim || victim->exec) victim = &r;
        } else if (!victim || (victim->exec && r.last_use < victim->last_use)) {
            victim = &r;
        }
    }
    const bool hit = found != nullptr;
    dlo_ctx::GraphRec& g = hit ? *found : *victim;
    g.last_use = ++c->graph_uses;
    LCHECK(cudaEventRecord(c->g_ev[0], c->xs), "event record");
    LCHECK(cudaStreamWaitEvent(c->cs, c->g_ev[0], 0), "join copy stream");
    if (hit) {
        // the graph's kernel event pairs hold its last launch until read
        if (g.tk_pending) collect_graph_timing(c, true);
        LCHECK(cudaGraphLaunch(g.exec, c->cs), "graph launch");
        g.tk_pending = !g.tk.empty();
        c->st.stagings += g.d_stagings;
        c->st.staged_bytes += g.d_staged_bytes;
        c->st.streamed_execs += g.d_streamed;
        c->st.kernel_launches += g.d_launches;
        c->st.h2d_copies += g.d_h2d;
        c->exec_counter += g.d_exec;
        for (size_t i = 0; i < g.lk.size(); ++i) c->log(g.lk[i], g.lb[i], g.ls[i]);
        c->slot_block[0] = g.slot_block_after[0];
        c->slot_block[1] = g.slot_block_after[1];
        ++c->st.graph_launches;
    } else {
        if (g.tk_pending) collect_graph_timing(c, true);
        if (g.exec) cudaGraphExecDestroy(g.exec);
        for (TimedKernel& t : g.tk) {
            cudaEventDestroy(t.a);
            cudaEventDestroy(t.b);
        }
        g = dlo_ctx::GraphRec();
        g.last_use = c->graph_uses;
        g.par = par;
        g.timing = c->timing;
        const HostSnap h0 = snap(c);
        const size_t k0 = c->kernels_pending.size();
        cudaError_t e = cudaStreamBeginCapture(c->cs, cudaStreamCaptureModeThreadLocal);
        if (e != cudaSuccess) return c->cuda_fail(e, "begin capture");
        c->capturing = true;
        c->cap_copy[0] = c->cap_copy[1] = c->cap_comp[0] = c->cap_comp[1] = false;
        // the copy stream joins the capture, and is joined back at its end
        e = cudaEventRecord(c->g_ev[1], c->cs);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(c->xs, c->g_ev[1], 0);
        dlo_status r = DLO_OK;
        if (e == cudaSuccess) {
            r = enqueue_forward(c, x_in, conds, ctx_tokens, batch, tokens, text_tokens, x_out);
            if (r == DLO_OK) {
                e = cudaEventRecord(c->g_ev[1], c->xs);
                if (e == cudaSuccess) e = cudaStreamWaitEvent(c->cs, c->g_ev[1], 0);
            }
        }
        c->capturing = false;
        cudaGraph_t graph = nullptr;
        const cudaError_t ee = cudaStreamEndCapture(c->cs, &graph);
        if (e == cudaSuccess) e = ee;
        cudaGraphExec_t exec = nullptr;
        if (r == DLO_OK && e == cudaSuccess) e = cudaGraphInstantiate(&exec, graph, 0);
        if (graph) cudaGraphDestroy(graph);
        if (r != DLO_OK || e != cudaSuccess) {
            // nothing captured ran: undo its host-side effects, turn graphs
            // off for this context and enqueue the forward directly
            cudaGetLastError();
            restore(c, h0);
            for (size_t i = k0; i < c->kernels_pending.size(); ++i) {
                c->ev_pool.push_back(c->kernels_pending[i].a);
                c->ev_pool.push_back(c->kernels_pending[i].b);
            }
            c->kernels_pending.resize(k0);
            if (r == DLO_OK) c->cuda_fail(e, "graph capture failed; graphs turned off");
            c->graphs = 0;
            c->drop_graphs();
            return enqueue_forward(c, x_in, conds, ctx_tokens, batch, tokens, text_tokens, x_out);
        }
        g.exec = exec;
        g.x_in = x_in;
        g.conds.assign(conds, conds + nc);
        g.ctx = ctx_tokens;
        g.x_out = x_out;
        g.B = batch;
        g.N = tokens;
        g.L = text_tokens;
        g.d_stagings = c->st.stagings - h0.st.stagings;
        g.d_staged_bytes = c->st.staged_bytes - h0.st.staged_bytes;
        g.d_streamed = c->st.streamed_execs - h0.st.streamed_execs;
        g.d_launches = c->st.kernel_launches - h0.st.kernel_launches;
        g.d_h2d = c->st.h2d_copies - h0.st.h2d_copies;
        g.d_exec = c->exec_counter - h0.exec;
        g.lk.assign(c->log_kind.begin() + h0.log_n, c->log_kind.end());
        g.lb.assign(c->log_block.begin() + h0.log_n, c->log_block.end());
        g.ls.assign(c->log_slot.begin() + h0.log_n, c->log_slot.end());
        g.slot_block_after[0] = c->slot_block[0];
        g.slot_block_after[1] = c->slot_block[1];
        // timing level 3: the captured event pairs now belong to the graph
        g.tk.assign(c->kernels_pending.begin() + k0, c->kernels_pending.end());
        c->kernels_pending.resize(k0);
        ++c->st.graph_captures;
        LCHECK(cudaGraphLaunch(g.exec, c->cs), "graph launch");
        g.tk_pending = !g.tk.empty();
        ++c->st.graph_launches;
    }
    for (int i = 0; i < 2; ++i) {
        LCHECK(cudaEventRecord(c->copy_done[i], c->cs), "event record");
        LCHECK(cudaEventRecord(c->compute_done[i], c->cs), "event record");
    }
    return DLO_OK;
}

}  // namespace

extern "C" dlo_status dlo_forward(dlo_ctx* c, const void* x_in, const void* cond,
                                  const void* ctx_tokens, int batch, int tokens, int text_tokens,
                                  void* x_out) {
    if (!c) return DLO_EINVAL;
    const Container& z = c->conts[0];
    for (const Container& k : c->conts)
        if (k.d.block_kind != z.d.block_kind || k.d.cond_dim != z.d.cond_dim)
            return c->fail(DLO_EINVAL, "containers take different conditionings: use dlo_forward_multi");
    std::vector<const void*> conds(c->conts.size(), cond);
    return forward_stack(c, x_in, conds.data(), ctx_tokens, batch, tokens, text_tokens, x_out);
}

extern "C" dlo_status dlo_forward_multi(dlo_ctx* c, const void* x_in, const void* const* conds,
                                        const void* ctx_tokens, int batch, int tokens, int text_tokens,
                                        void* x_out) {
    if (!c) return DLO_EINVAL;
    if (!conds) return c->fail(DLO_EINVAL, "conds is NULL");
    return forward_stack(c, x_in, conds, ctx_tokens, batch, tokens, text_tokens, x_out);
}

extern "C" dlo_status dlo_wait(dlo_ctx* c, int timeout_ms) {
    if (!c) return DLO_EINVAL;
    if (timeout_ms <= 0) timeout_ms = 60000;
    cudaSetDevice(c->device);
    cudaError_t e = cudaSuccess;
    if (!stream_wait(c->cs, timeout_ms, &e) || !stream_wait(c->xs, timeout_ms, &e)) {
        if (e == cudaErrorNotReady) return c->fail(DLO_ETIMEDOUT, "streams still busy after %d ms", timeout_ms);
        return c->cuda_fail(e, "stream query");
    }
    return check_device_error(c);
}

extern "C" dlo_status dlo_forward_host(dlo_ctx* c, const void* x_in, const void* cond,
                                       const void* ctx_tokens, int batch, int tokens,
                                       int text_tokens, void* x_out, int timeout_ms) {
    if (!c) return DLO_EINVAL;
    if (c->state != kRegistered) return c->fail(DLO_ESTATE, "register host blocks first");
    if (c->conts.size() != 1)
        return c->fail(DLO_EUNSUPPORTED, "host-buffer forward takes single-container stacks");
    const dlo_desc& d = c->d;
    if (d.block_kind == DLO_BLOCK_BYTES) {
        if (!x_out) return c->fail(DLO_EINVAL, "NULL output");
        cudaSetDevice(c->device);
        void* sums = c->wsp + c->ws.in_x;
        dlo_status r = dlo_forward(c, nullptr, nullptr, nullptr, 1, 1, 0, sums);
        if (r != DLO_OK) return r;
        LCHECK(cudaMemcpyAsync(x_out, sums, static_cast<size_t>(d.n_blocks) * 8, cudaMemcpyDeviceToHost, c->cs),
               "D2H checksums");
        return dlo_wait(c, timeout_ms);
    }
    if (batch < 1 || batch > d.max_batch || tokens < 1 || tokens > d.max_tokens)
        return c->fail(DLO_EINVAL, "batch/tokens out of range");
    if (!x_in || !x_out || !cond) return c->fail(DLO_EINVAL, "NULL input/output");
    if (d.block_kind == DLO_BLOCK_VIDEO &&
        (!ctx_tokens || text_tokens < 1 || text_tokens > d.max_text_tokens))
        return c->fail(DLO_EINVAL, "ctx_tokens/text_tokens invalid");
    cudaSetDevice(c->device);
    const size_t xb = static_cast<size_t>(batch) * tokens * d.hidden * 2;
    void* dx = c->wsp + c->ws.in_x;
    void* dc = c->wsp + c->ws.in_cond;
    void* dt = d.block_kind == DLO_BLOCK_VIDEO ? c->wsp + c->ws.in_ctx : nullptr;
    const size_t cb = d.block_kind == DLO_BLOCK_DIT ? static_cast<size_t>(batch) * d.cond_dim * 2
                                                    : static_cast<size_t>(batch) * 6 * d.hidden * 4;
    LCHECK(cudaMemcpyAsync(dx, x_in, xb, cudaMemcpyHostToDevice, c->cs), "H2D x");
    LCHECK(cudaMemcpyAsync(dc, cond, cb, cudaMemcpyHostToDevice, c->cs), "H2D cond");
    if (dt)
        LCHECK(cudaMemcpyAsync(dt, ctx_tokens, static_cast<size_t>(batch) * text_tokens * d.text_dim * 2,
                               cudaMemcpyHostToDevice, c->cs),
               "H2D ctx");
    dlo_status r = dlo_forward(c, dx, dc, dt, batch, tokens, text_tokens, dx);
    if (r != DLO_OK) return r;
    LCHECK(cudaMemcpyAsync(x_out, dx, xb, cudaMemcpyDeviceToHost, c->cs), "D2H x");
    return dlo_wait(c, timeout_ms);
}

extern "C" dlo_status dlo_destroy(dlo_ctx* c) {
    if (!c) return DLO_OK;
    cudaSetDevice(c->device);
    dlo_status first = DLO_OK;
    cudaError_t e = cudaSuccess;
    const bool idle = stream_wait(c->cs, 60000, &e) && stream_wait(c->xs, 60000, &e);
    if (!idle) first = DLO_ETIMEDOUT;
    if (idle) {
        // unregister only after the device no longer reads the ranges
        for (auto& u : c->reg_ranges) {
            if (cudaHostUnregister(u.first) != cudaSuccess) {
                cudaGetLastError();
                if (first == DLO_OK) first = DLO_EREGISTER;
            }
        }
    }
    for (int i = 0; i < 2; ++i) {
        if (c->copy_done[i]) cudaEventDestroy(c->copy_done[i]);
        if (c->compute_done[i]) cudaEventDestroy(c->compute_done[i]);
    }
    if (c->resident_ev) cudaEventDestroy(c->resident_ev);
    c->drop_graphs();
    for (int i = 0; i < 2; ++i)
        if (c->g_ev[i]) cudaEventDestroy(c->g_ev[i]);
    for (auto& t : c->timed_pending)
        for (cudaEvent_t ev : {t.copy0, t.copy1, t.wait0, t.comp0, t.comp1}) cudaEventDestroy(ev);
    for (auto& t : c->kernels_pending) {
        cudaEventDestroy(t.a);
        cudaEventDestroy(t.b);
    }
    for (cudaEvent_t ev : c->ev_pool) cudaEventDestroy(ev);
    if (idle) {
        for (int i = 0; i < 2; ++i)
            if (c->hstage[i]) cudaFreeHost(c->hstage[i]);
    }
    c->packer.reset();
    delete c;
    return first;
}

extern "C" dlo_status dlo_get_stats(dlo_ctx* c, dlo_stats* out) {
    if (!c || !out) return DLO_EINVAL;
    cudaSetDevice(c->device);
    collect_timing(c);
    c->st.slot_block[0] = c->slot_block[0];
    c->st.slot_block[1] = c->slot_block[1];
    c->st.registered_ranges = static_cast<int>(c->reg_ranges.size());
    c->st.registered_read_only = c->reg_read_only ? 1 : 0;
    *out = c->st;
    return DLO_OK;
}

extern "C" dlo_status dlo_get_log(dlo_ctx* c, int* kind, int* block, int* slot, int cap, int* count) {
    if (!c) return DLO_EINVAL;
    if (count) *count = static_cast<int>(c->log_total);
    const int n = std::min<int>(cap, static_cast<int>(c->log_kind.size()));
    for (int i = 0; i < n; ++i) {
        if (kind) kind[i] = c->log_kind[i];
        if (block) block[i] = c->log_block[i];
        if (slot) slot[i] = c->log_slot[i];
    }
    return DLO_OK;
}

extern "C" dlo_status dlo_reset_log(dlo_ctx* c) {
    if (!c) return DLO_EINVAL;
    c->log_kind.clear();
    c->log_block.clear();
    c->log_slot.clear();
    c->log_total = 0;
    return DLO_OK;
}

extern "C" dlo_status dlo_set_graphs(dlo_ctx* c, int on) {
    if (!c) return DLO_EINVAL;
    if (on != 0 && on != 1) return c->fail(DLO_EINVAL, "graphs must be 0 or 1");
    cudaSetDevice(c->device);
    if (!on) c->drop_graphs();
    c->graphs = on;
    return DLO_OK;
}

extern "C" dlo_status dlo_set_timing(dlo_ctx* c, int on) {
    if (!c) return DLO_EINVAL;
    if (on < 0 || on > 3) return c->fail(DLO_EINVAL, "timing level must be 0, 1, 2 or 3");
    c->timing = on;
    return DLO_OK;
}

extern "C" dlo_status dlo_verify_slot(dlo_ctx* c, int slot, int block) {
    if (!c) return DLO_EINVAL;
    if (slot < 0 || slot > 1) return c->fail(DLO_EINVAL, "slot must be 0 or 1");
    if (c->state != kRegistered) return c->fail(DLO_ESTATE, "no host blocks attached");
    if (block < 0) block = c->slot_block[slot];
    if (block < 0 || block >= c->d.n_blocks) return c->fail(DLO_EINVAL, "no block staged in slot %d", slot);
    cudaSetDevice(c->device);
    cudaError_t e = cudaSuccess;
    if (!stream_wait(c->xs, 60000, &e)) return c->fail(DLO_ETIMEDOUT, "copy stream busy");
    const size_t nb = c->bytes_of(block);
    std::vector<uint8_t> tmp(nb);
    e = cudaMemcpy(tmp.data(), c->slot[slot], nb, cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return c->cuda_fail(e, "slot read-back");
    if (std::memcmp(tmp.data(), c->host[block], nb) != 0)
        return c->fail(DLO_EMISMATCH, "slot %d differs from host block %d", slot, block);
    return DLO_OK;
}

// ===================================================================== unit ops

namespace {
unsigned long long g_op_launches = 0;
}  // namespace

namespace dlo {

dlo_status op_fail(dlo_status st, const std::string& msg) {
    g_create_error = msg;
    return st;
}

dlo_status op_result(cudaError_t e) {
    if (e == cudaSuccess) return DLO_OK;
    cudaGetLastError();
    return op_fail(DLO_ECUDA, std::string("kernel launch: ") + cudaGetErrorString(e));
}

}  // namespace dlo

namespace {
dlo_status op_inval(const char* m) { return op_fail(DLO_EINVAL, m); }
}  // namespace

extern "C" dlo_status dlo_op_wait_selftest(int* err, void* stream) {
    if (!err || !aligned(err, 4)) return op_inval("err must be a 4-byte aligned device int");
    return op_result(launch_wait_selftest(err, static_cast<cudaStream_t>(stream), &g_op_launches));
}

extern "C" dlo_status dlo_debug_device_timeout(dlo_ctx* c) {
    if (!c) return DLO_EINVAL;
    cudaSetDevice(c->device);
    return c->timed(DLO_K_CONVERT, 0.0, 0.0, c->cs, [&] {
               return launch_wait_selftest(c->err_word(), c->cs, &c->st.kernel_launches);
           }) == cudaSuccess
               ? DLO_OK
               : c->fail(DLO_ECUDA, "launch of the wait self-test failed");
}

extern "C" dlo_status dlo_op_quantize_act(const void* x, int rows, int cols, int ld, void* q, float* scale,
                                          float* scratch, void* stream) {
    if (!x || !q || !scale || !scratch) return op_inval("NULL argument");
    if (rows < 1 || cols < 8 || cols % 8 || ld < cols || ld % 8) return op_inval("need cols % 8 == 0, ld >= cols, ld % 8 == 0");
    if (!aligned(x, 16) || !aligned(q, 16) || !aligned(scale, 4) || !aligned(scratch, 4))
        return op_inval("x and q must be 16-byte aligned");
    return op_result(launch_quantize_e4m3(x, rows, cols, ld, q, scale, scratch, static_cast<cudaStream_t>(stream),
                                          &g_op_launches));
}

extern "C" dlo_status dlo_op_gemm_w8a8(const void* A, const float* a_scale, const void* W, const float* scales,
                                       int scale_seg, const void* bias, int M, int N, int K, int epilogue,
                                       void* out, int ldo, const float* gate, int gate_ld, int rows_per_batch,
                                       int* err, void* stream) {
    if (!a_scale || !scales) return op_inval("W8A8 needs the activation scale and the weight scales");
    if (!aligned(a_scale, 4)) return op_inval("a_scale misaligned");
    GemmParams p;
    dlo_status r = op_gemm_params(A, W, DLO_DT_E4M3, scales, scale_seg, bias, M, N, K, epilogue, out, ldo, gate,
                                  gate_ld, rows_per_batch, DLO_DT_E4M3, a_scale, &p);
    if (r != DLO_OK) return r;
    p.err = err;
    return op_launch_gemm(p, static_cast<cudaStream_t>(stream));
}

extern "C" dlo_status dlo_op_gemm(const void* A, const void* W, int w_dtype, const float* scales,
                                  int scale_seg, const void* bias, int M, int N, int K, int epilogue,
                                  void* out, int ldo, const float* gate, int gate_ld,
                                  int rows_per_batch, int* err, void* stream) {
    GemmParams p;
    dlo_status r = op_gemm_params(A, W, w_dtype, scales, scale_seg, bias, M, N, K, epilogue, out, ldo, gate,
                                  gate_ld, rows_per_batch, DLO_DT_BF16, nullptr, &p);
    if (r != DLO_OK) return r;
    p.err = err;
    return op_launch_gemm(p, static_cast<cudaStream_t>(stream));
}

namespace dlo {

dlo_status op_gemm_params(const void* A, const void* W, int w_dtype, const float* scales, int scale_seg,
                          const void* bias, int M, int N, int K, int epilogue, void* out, int ldo,
                          const float* gate, int gate_ld, int rows_per_batch, int a_dtype,
                          const float* a_scale, GemmParams* p) {
    if (!A || !W || !out) return op_inval("NULL operand");
    if (M < 1 || N < 16 || N % 16 || K < 16 || K % 16) return op_inval("need M >= 1, N % 16 == 0, K % 16 == 0");
    if (!aligned(A, 16) || !aligned(W, 16) || !aligned(out, 16) || ldo % 8 || ldo < N)
        return op_inval("operands must be 16-byte aligned and ldo % 8 == 0, ldo >= N");
    if (w_dtype != DLO_DT_BF16 && w_dtype != DLO_DT_E4M3) return op_inval("w_dtype");
    if (epilogue < DLO_EPI_BIAS || epilogue > DLO_EPI_RESIDUAL) return op_inval("epilogue");
    if (scales && (scale_seg < 16 || scale_seg % 16)) return op_inval("scale_seg % 16 != 0");
    if (bias && !aligned(bias, 16)) return op_inval("bias must be 16-byte aligned");
    if (gate && (!aligned(gate, 16) || gate_ld % 4 || rows_per_batch < 1)) return op_inval("gate layout");
    GemmParams q;
    q.A = A;
    q.W = W;
    q.w_dtype = w_dtype;
    q.scales = scales;
    q.scale_seg = scale_seg;
    q.bias = bias;
    q.M = M;
    q.N = N;
    q.K = K;
    q.epi = epilogue;
    q.out = out;
    q.ldo = ldo;
    q.gate = gate;
    q.gate_ld = gate_ld;
    q.rows_per_batch = rows_per_batch > 0 ? rows_per_batch : 1;
    q.a_dtype = a_dtype;
    q.a_scale = a_scale;
    *p = q;
    return DLO_OK;
}

dlo_status op_launch_gemm(const GemmParams& p, cudaStream_t s) {
    return op_result(launch_gemm(p, s, &g_op_launches));
}

}  // namespace dlo

extern "C" dlo_status dlo_op_attention(const void* Q, const void* K, const void* V, void* O, int batch,
                                       int heads, int head_dim, int nq, int nk, int ldq, int ldk, int ldv,
                                       int ldo, void* stream) {
    if (!Q || !K || !V || !O) return op_inval("NULL operand");
    if (batch < 1 || heads < 1 || nq < 1 || nk < 1) return op_inval("sizes must be >= 1");
    if (head_dim < 8 || head_dim % 8 || head_dim > 128) return op_inval("head_dim % 8 != 0 or > 128");
    if (ldq % 8 || ldk % 8 || ldv % 8 || ldo % 8) return op_inval("ld % 8 != 0");
    if (!aligned(Q, 16) || !aligned(K, 16) || !aligned(V, 16) || !aligned(O, 16)) return op_inval("alignment");
    return op_result(launch_attention(Q, K, V, O, batch, heads, head_dim, nq, nk, ldq, ldk, ldv, ldo,
                                      nullptr, static_cast<cudaStream_t>(stream), &g_op_launches));
}

extern "C" dlo_status dlo_op_layernorm(const float* x, int rows, int D, int rows_per_batch,
                                       const float* shift, const float* scale, int mod_ld, const void* w,
                                       const void* b, float eps, void* out, void* stream) {
    if (!x || !out || rows < 1 || D < 4 || D % 4 || rows_per_batch < 1) return op_inval("layernorm args");
    if ((shift == nullptr) != (scale == nullptr) || (w == nullptr) != (b == nullptr)) return op_inval("pairs");
    if (scale && (mod_ld % 4 || !aligned(scale, 16) || !aligned(shift, 16))) return op_inval("mod layout");
    return op_result(launch_layernorm(x, rows, D, rows_per_batch, shift, scale, mod_ld, w, b, eps, out,
                                      static_cast<cudaStream_t>(stream), &g_op_launches));
}

extern "C" dlo_status dlo_op_rmsnorm(void* x, int rows, int D, int ld, int col0, const void* w, float eps,
                                     void* stream) {
    if (!x || !w || rows < 1 || D < 8 || D % 8 || ld % 8 || col0 % 8 || col0 + D > ld) return op_inval("rmsnorm args");
    return op_result(launch_rmsnorm(x, rows, D, ld, col0, w, eps, static_cast<cudaStream_t>(stream), &g_op_launches));
}

extern "C" dlo_status dlo_op_adaln(const void* cvec, int B, int C, const void* W, const void* bias, int N,
                                   float* m, void* stream) {
    if (!cvec || !W || !bias || !m || B < 1 || C < 8 || C % 8 || N < 1) return op_inval("adaln args");
    return op_result(launch_adaln(cvec, B, C, W, bias, N, m, static_cast<cudaStream_t>(stream), &g_op_launches));
}

extern "C" dlo_status dlo_op_stage(void* dst, const void* src, size_t bytes, int mode, void* stream) {
    if (!dst || !src || bytes % 16 || !aligned(dst, 16) || !aligned(src, 16)) return op_inval("stage args");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (mode == DLO_STAGE_GATHER) return op_result(launch_gather(dst, src, bytes, s, &g_op_launches));
    if (mode == DLO_STAGE_MEMCPY) return op_result(cudaMemcpyAsync(dst, src, bytes, cudaMemcpyDefault, s));
    return op_inval("mode");
}
