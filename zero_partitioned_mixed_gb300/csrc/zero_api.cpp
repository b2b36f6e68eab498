// Host side of the C ABI declared in include/zero_gb300.h: argument
// validation, the flat partition, exact accounting, workspace ownership and
// the order of kernel launches for each stage and mode.  Nothing here waits
// on the device except zero_get_status and zero_destroy.

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <new>
#include <string>
#include <utility>
#include <vector>

#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>

#include "zero_gb300.h"
#include "zero_internal.h"

namespace {

thread_local std::string g_init_error;

// An NVTX range over one call of the C ABI, so that a profiler's timeline
// shows which entry point issued which kernels (header-only NVTX 3: no
// cost unless a tool is attached).
struct CallRange {
    explicit CallRange(const char* name) { nvtxRangePushA(name); }
    ~CallRange() { nvtxRangePop(); }
    CallRange(const CallRange&) = delete;
    CallRange& operator=(const CallRange&) = delete;
};

}  // namespace

struct zero_handle {
    uint64_t psi = 0, psi_pad = 0, shard = 0;
    int n = 0, stage = 0, dtype = 0, align = 0;
    unsigned flags = 0;
    int device = 0;
    std::vector<uint64_t> offsets, real;
    zg::Workspace ws{};
    void* ws_block = nullptr;
    // ZeRO-3 step bookkeeping (host side)
    std::vector<std::pair<uint64_t, uint64_t>> covered;
    int rs_calls = 0;
    int rs_mode = -1;
    zero_hyper_t rs_hyper{};
    // accounting
    uint64_t last_r = 0, last_w = 0, tot_r = 0, tot_w = 0;
    uint64_t persist_from = 0;   // stage 3: start of the resident region (psi_pad = none)
    uint64_t hold_tile1 = 0;   // zero_debug_hold_staged, for the next staged step
    uint64_t launch_seq = 0;   // chunked launches: counter slot = launch_seq % kCtrSlots
    std::string err;
};

namespace {

int fail(zero_handle* h, int code, const std::string& msg) {
    if (h) h->err = msg;
    else g_init_error = msg;
    return code;
}

int cuda_fail(zero_handle* h, cudaError_t e, const char* what) {
    return fail(h, ZERO_ECUDA, std::string(what) + ": " + cudaGetErrorString(e));
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool double_buffered(const zero_handle* h) { return (h->flags & ZERO_F_DOUBLE_BUFFER) != 0; }

void count(zero_handle* h, uint64_t r, uint64_t w) {
    h->last_r = r;
    h->last_w = w;
    h->tot_r += r;
    h->tot_w += w;
}

// Resolve AUTO and check that the requested mode fits the handle.  A
// one-shot step (stages 1/2 with all gradients at hand) can be speculative
// even with clipping: when the norm calls for clipping it is redone from the
// old slot.  Bucketed steps release each bucket's gradients, so clipping
// there needs the two-pass mode.
int resolve_mode(zero_handle* h, const zero_hyper_t* hy, int* mode, bool one_shot = false) {
    const bool clip = hy->max_norm > 0.0f && !one_shot;
    const bool db = double_buffered(h);
    switch (hy->mode) {
        case ZERO_MODE_AUTO:
            if (h->stage != 0 && db && !clip) *mode = ZERO_MODE_SPECULATIVE;
            else if (h->stage == 0 || h->stage == 3) *mode = ZERO_MODE_TWO_PASS_WS;
            else *mode = h->n > 4 ? ZERO_MODE_TWO_PASS_WS : ZERO_MODE_TWO_PASS_REREAD;
            return ZERO_OK;
        case ZERO_MODE_SPECULATIVE:
            if (h->stage == 0) return fail(h, ZERO_EINVAL, "speculative mode is not available for stage 0");
            if (!db) return fail(h, ZERO_EINVAL, "speculative mode needs ZERO_F_DOUBLE_BUFFER state");
            if (clip)
                return fail(h, ZERO_EINVAL,
                            "clipping a bucketed step needs the global norm before the update: use a two-pass mode");
            *mode = ZERO_MODE_SPECULATIVE;
            return ZERO_OK;
        case ZERO_MODE_SPECULATIVE_STAGED:
            if (!one_shot || h->stage == 0 || h->stage == 3)
                return fail(h, ZERO_EINVAL, "staged speculative mode is for the one-shot stage 1/2 step");
            if (!db) return fail(h, ZERO_EINVAL, "speculative mode needs ZERO_F_DOUBLE_BUFFER state");
            if (zg::tma_stages(h->n) < 2) return fail(h, ZERO_EINVAL, "staged mode supports up to 19 ranks");
            if (h->psi_pad % 8) return fail(h, ZERO_EINVAL, "staged mode needs psi_pad to be a multiple of 8");
            *mode = ZERO_MODE_SPECULATIVE_STAGED;
            return ZERO_OK;
        case ZERO_MODE_TWO_PASS_WS:
            *mode = ZERO_MODE_TWO_PASS_WS;
            return ZERO_OK;
        case ZERO_MODE_TWO_PASS_REREAD:
            if (h->stage == 0 || h->stage == 3)
                return fail(h, ZERO_EINVAL, "stages 0 and 3 keep g_hat in the workspace: use TWO_PASS_WS or AUTO");
            *mode = ZERO_MODE_TWO_PASS_REREAD;
            return ZERO_OK;
        default:
            return fail(h, ZERO_EINVAL, "unknown mode");
    }
}

int ensure_ghat(zero_handle* h) {
    if (h->ws.ghat || h->psi_pad == 0) return ZERO_OK;
    void* p = nullptr;
    cudaError_t e = cudaMalloc(&p, h->psi_pad * sizeof(float));
    if (e != cudaSuccess) {
        cudaGetLastError();
        return fail(h, ZERO_ENOMEM, "cannot allocate the fp32 gradient workspace (" +
                                        std::to_string(h->psi_pad * 4) + " bytes)");
    }
    h->ws.ghat = static_cast<float*>(p);
    return ZERO_OK;
}

zg::Args base_args(const zero_handle* h, const zero_hyper_t* hy) {
    zg::Args a;
    std::memset(&a, 0, sizeof(a));
    a.n_ranks = h->n;
    a.stage = h->stage;
    a.psi = h->psi;
    a.psi_pad = h->psi_pad;
    a.ws = h->ws;
    if (hy) {
        a.hyper.lr = hy->lr;
        a.hyper.beta1 = hy->beta1;
        a.hyper.beta2 = hy->beta2;
        a.hyper.eps = hy->eps;
        a.hyper.weight_decay = hy->weight_decay;
        a.hyper.max_norm = hy->max_norm;
    }
    return a;
}

bool aligned32(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 31u) == 0; }

// 8-wide launches use 256-bit fp32 accesses when every fp32 buffer of the
// launch is 32-byte aligned (slot and replica strides are multiples of 8
// floats whenever the 8-wide path runs), else 128-bit ones.
zg::Vec pick_vec(bool vec8, const zg::Args& a) {
    if (!vec8) return zg::Vec::k1;
    const bool s32 = aligned32(a.master) && aligned32(a.m) && aligned32(a.v) && aligned32(a.ws.ghat);
    return s32 ? zg::Vec::k8s32 : zg::Vec::k8s16;
}

// The 8-wide path of a bucket [a0, a0 + L) that touches the fp32 state: the
// bucket on 8-element boundaries, and with two state slots the second slot's
// base (psi_pad floats in) on one too, else its vector accesses would be
// misaligned.
bool bucket_vec8(const zero_handle* h, uint64_t a0, uint64_t L) {
    return (a0 % 8) == 0 && (L % 8) == 0 && (!double_buffered(h) || (h->psi_pad % 8) == 0);
}

// Each chunked launch its own counter slot: a gather on one stream may
// overlap a reduce-scatter on another.
int next_slot(zero_handle* h) { return static_cast<int>(h->launch_seq++ % zg::kCtrSlots); }

int launch(zero_handle* h, zg::Kind kind, bool vec8, const zg::Args& a, cudaStream_t s, const char* what) {
    zg::Args b = a;
    b.ctr_slot = next_slot(h);
    cudaError_t e = zg::launch(kind, h->dtype, pick_vec(vec8, b), b, s, nullptr);
    if (e != cudaSuccess) return cuda_fail(h, e, what);
    return ZERO_OK;
}

int check_ptr(zero_handle* h, const void* p, const char* name) {
    if (!p) return fail(h, ZERO_EINVAL, std::string(name) + " is NULL");
    if (!aligned16(p)) return fail(h, ZERO_EINVAL, std::string(name) + " is not 16-byte aligned");
    return ZERO_OK;
}

int check_hyper(zero_handle* h, const zero_hyper_t* hy) {
    if (!hy) return fail(h, ZERO_EINVAL, "hyper is NULL");
    const float vals[] = {hy->lr, hy->beta1, hy->beta2, hy->eps, hy->weight_decay, hy->max_norm};
    for (float x : vals)
        if (!std::isfinite(x)) return fail(h, ZERO_EINVAL, "hyper-parameters must be finite");
    if (!(hy->beta1 >= 0.0f && hy->beta1 < 1.0f && hy->beta2 >= 0.0f && hy->beta2 < 1.0f))
        return fail(h, ZERO_EINVAL, "beta1 and beta2 must lie in [0, 1)");
    return ZERO_OK;
}

bool same_hyper(const zero_hyper_t& x, const zero_hyper_t& y) {
    return std::memcmp(&x, &y, sizeof(zero_hyper_t)) == 0;
}

// Reduce-scatter of one bucket of a step whose gradients arrive bucket by
// bucket (stage 3 always; stage 2 when the caller reduces during backward).
// outs: the 16-bit shard (stage 3) or the N replicas (stage 2).
// gout (stage 3, 8-wide, checked by the caller): the same launch then
// gathers [ga, ga + gcount) of the shard outs[0] into gout[r].
int rs_bucket(zero_handle* h, uint64_t a0, uint64_t b0, const void* const* grads, float* master, float* m,
              float* v, void* const* outs, const zero_hyper_t* hyper, void* stream, int qbits = 0,
              const float* const* qscales = nullptr, uint64_t ga = 0, uint64_t gcount = 0,
              void* const* gout = nullptr) {
    int rc = check_hyper(h, hyper);
    if (rc) return rc;
    if (a0 > b0 || b0 > h->psi_pad) return fail(h, ZERO_EINVAL, "bucket must satisfy 0 <= a <= b <= psi_pad");
    const uint64_t L = b0 - a0, N = static_cast<uint64_t>(h->n);
    for (auto& iv : h->covered)
        if (a0 < iv.second && iv.first < b0)
            return fail(h, ZERO_ESTATE, "bucket overlaps one already reduced this step");
    if (h->rs_calls >= zg::kMaxBuckets) return fail(h, ZERO_ESTATE, "more than 4096 buckets in one step");
    int mode = 0;
    if (h->rs_calls == 0) {
        if ((rc = resolve_mode(h, hyper, &mode))) return rc;
        // the gradients are gone once their bucket is reduced: no re-read pass
        if (mode == ZERO_MODE_TWO_PASS_REREAD) {
            if (hyper->mode == ZERO_MODE_TWO_PASS_REREAD)
                return fail(h, ZERO_EINVAL, "bucketed reduce-scatter keeps g_hat in the workspace: no REREAD mode");
            mode = ZERO_MODE_TWO_PASS_WS;
        }
    } else {
        if (!same_hyper(*hyper, h->rs_hyper))
            return fail(h, ZERO_EINVAL, "every reduce-scatter of one step must pass the same hyper");
        mode = h->rs_mode;
    }
    if (L == 0) {
        count(h, 0, 0);
        return ZERO_OK;
    }
    if (!grads) return fail(h, ZERO_EINVAL, "grads is NULL");
    zg::Args a = base_args(h, hyper);
    for (int r = 0; r < h->n; ++r) {
        if ((rc = check_ptr(h, grads[r], qbits ? "codes[r]" : "grads[r]"))) return rc;
        a.grads[r] = grads[r];
        if (qbits) {
            if (!qscales || !qscales[r] || (reinterpret_cast<uintptr_t>(qscales[r]) & 7u))
                return fail(h, ZERO_EINVAL, "scales[r] is NULL or not 8-byte aligned");
            a.qsrc[r] = qscales[r];
        }
    }
    a.qbits = qbits;
    const bool spec = mode == ZERO_MODE_SPECULATIVE;
    const int n_out = h->stage == 3 ? 1 : h->n;
    if (spec) {
        if ((rc = check_ptr(h, master, "master")) || (rc = check_ptr(h, m, "m")) || (rc = check_ptr(h, v, "v")))
            return rc;
        if (!outs) return fail(h, ZERO_EINVAL, "params is NULL");
        for (int r = 0; r < n_out; ++r) {
            if ((rc = check_ptr(h, outs[r], h->stage == 3 ? "shard16" : "params[r]"))) return rc;
            a.params[r] = outs[r];
        }
    } else {
        if ((rc = ensure_ghat(h))) return rc;
    }
    a.master = master;
    a.m = m;
    a.v = v;
    a.ws = h->ws;
    a.slot_stride = double_buffered(h) ? h->psi_pad : 0;
    a.base = a0;
    a.count = L;
    a.bucket_index = h->rs_calls;
    const bool vec8 = bucket_vec8(h, a0, L);
    if (qbits) {
        const cudaError_t e = zg::launch_q(spec ? zg::QKind::kRsQSpec : zg::QKind::kRsQWs, h->dtype, qbits,
                                           pick_vec(vec8, a), a, static_cast<cudaStream_t>(stream));
        if (e != cudaSuccess) return cuda_fail(h, e, "quantized reduce-scatter");
    } else if (gout) {
        a.params[0] = outs[0];   // the gather's source, also in two-pass mode
        for (int r = 0; r < h->n; ++r) a.gout[r] = gout[r];
        a.gbase = ga;
        a.gcount = gcount;
        const zg::Kind kind = spec ? zg::Kind::kRsSpecGather : zg::Kind::kRsWsGather;
        if ((rc = launch(h, kind, vec8, a, static_cast<cudaStream_t>(stream), "reduce-scatter + gather"))) return rc;
    } else {
        const zg::Kind kind =
            !spec ? zg::Kind::kRsWs : (h->stage == 3 ? zg::Kind::kRsSpec : zg::Kind::kRsSpecReplicas);
        if ((rc = launch(h, kind, vec8, a, static_cast<cudaStream_t>(stream), "reduce-scatter"))) return rc;
    }
    if (h->rs_calls == 0) {
        h->rs_mode = mode;
        h->rs_hyper = *hyper;
    }
    h->rs_calls += 1;
    h->covered.emplace_back(a0, b0);
    const uint64_t in_bytes = qbits ? N * (L * qbits / 8 + 8 * ((L + zg::kQBlock - 1) / zg::kQBlock)) : 2 * N * L;
    const uint64_t g_r = gout ? 2 * gcount : 0, g_w = gout ? 2 * N * gcount : 0;
    if (spec) count(h, in_bytes + 12 * L + g_r, 12 * L + 2 * static_cast<uint64_t>(n_out) * L + g_w);
    else count(h, in_bytes + g_r, 4 * L + g_w);
    return ZERO_OK;
}

// Byte ranges [p, p + n) and [q, q + k) share a byte.
bool overlaps(const void* p, uint64_t n, const void* q, uint64_t k) {
    const uintptr_t a = reinterpret_cast<uintptr_t>(p), b = reinterpret_cast<uintptr_t>(q);
    return n > 0 && k > 0 && a < b + k && b < a + n;
}

bool aligned8(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 7u) == 0; }

}  // namespace

void zg::set_global_error(const char* msg) { g_init_error = msg ? msg : ""; }

extern "C" {

int zero_init_partition(uint64_t psi, int n_ranks, int stage, int dtype, int align, unsigned flags,
                        zero_handle_t* out) {
    if (!out) return fail(nullptr, ZERO_EINVAL, "out is NULL");
    *out = nullptr;
    if (n_ranks < 1 || n_ranks > ZERO_MAX_RANKS)
        return fail(nullptr, ZERO_EINVAL, "n_ranks must be in 1..64");
    if (stage < 0 || stage > 3) return fail(nullptr, ZERO_EINVAL, "stage must be 0..3");
    if (dtype != ZERO_FP16 && dtype != ZERO_BF16) return fail(nullptr, ZERO_EINVAL, "dtype must be fp16 or bf16");
    if (align < 1) return fail(nullptr, ZERO_EINVAL, "align must be >= 1");
    if (flags & ~ZERO_F_DOUBLE_BUFFER) return fail(nullptr, ZERO_EINVAL, "unknown flag");
    if (stage == 0 && (flags & ZERO_F_DOUBLE_BUFFER))
        return fail(nullptr, ZERO_EINVAL, "stage 0 keeps its state in place (no double buffer)");
    const uint64_t unit = static_cast<uint64_t>(n_ranks) * static_cast<uint64_t>(align);
    if (psi > (UINT64_MAX / 64) - unit) return fail(nullptr, ZERO_EINVAL, "psi too large");

    zero_handle* h = new (std::nothrow) zero_handle();
    if (!h) return fail(nullptr, ZERO_ENOMEM, "host allocation failed");
    h->psi = psi;
    h->n = n_ranks;
    h->stage = stage;
    h->dtype = dtype;
    h->align = align;
    h->flags = flags;
    h->psi_pad = (psi + unit - 1) / unit * unit;
    h->shard = h->psi_pad / static_cast<uint64_t>(n_ranks);
    h->persist_from = h->psi_pad;
    for (int r = 0; r < n_ranks; ++r) {
        const uint64_t off = static_cast<uint64_t>(r) * h->shard;
        h->offsets.push_back(off);
        h->real.push_back(psi > off ? std::min(psi - off, h->shard) : 0);
    }
    cudaError_t e = cudaGetDevice(&h->device);
    if (e != cudaSuccess) {
        delete h;
        return cuda_fail(nullptr, e, "cudaGetDevice");
    }
    // one block: status | partials | bucket partials | flags | bucket flags |
    // chunk counters | group tickets | chunk partials | group partials
    const size_t st_bytes = (sizeof(zg::DevStatus) + 255) / 256 * 256;
    auto r256 = [](size_t x) { return (x + 255) / 256 * 256; };
    const size_t fixed = r256(zg::kMaxBlocks * (sizeof(double) + sizeof(int32_t)) +
                              zg::kMaxBuckets * (sizeof(double) + sizeof(int32_t)));
    const uint64_t nch = zg::max_chunks(h->psi_pad), ngr = zg::max_groups(h->psi_pad);
    const size_t ctr_bytes = r256(zg::kCtrSlots * sizeof(zg::ChunkCtr));
    const size_t tk_bytes = r256(ngr * sizeof(uint32_t));
    const size_t cp_bytes = r256(nch * sizeof(double));
    const size_t gp_bytes = r256(ngr * sizeof(double));
    const size_t bytes = st_bytes + fixed + ctr_bytes + tk_bytes + cp_bytes + gp_bytes;
    e = cudaMalloc(&h->ws_block, bytes);
    if (e != cudaSuccess) {
        cudaGetLastError();
        delete h;
        return fail(nullptr, ZERO_ENOMEM, "cannot allocate the workspace");
    }
    char* base = static_cast<char*>(h->ws_block);
    h->ws.status = reinterpret_cast<zg::DevStatus*>(base);
    h->ws.partials = reinterpret_cast<double*>(base + st_bytes);
    h->ws.bucket_norm = h->ws.partials + zg::kMaxBlocks;
    h->ws.flags = reinterpret_cast<int32_t*>(h->ws.bucket_norm + zg::kMaxBuckets);
    h->ws.bucket_flag = h->ws.flags + zg::kMaxBlocks;
    h->ws.ghat = nullptr;
    char* sched = base + st_bytes + fixed;
    h->ws.ctrs = reinterpret_cast<zg::ChunkCtr*>(sched);
    h->ws.group_ticket = reinterpret_cast<uint32_t*>(sched + ctr_bytes);
    h->ws.chunk_part = reinterpret_cast<double*>(sched + ctr_bytes + tk_bytes);
    h->ws.group_part = reinterpret_cast<double*>(sched + ctr_bytes + tk_bytes + cp_bytes);
    e = cudaMemset(h->ws_block, 0, bytes);
    if (e == cudaSuccess) e = zg::launch_set_scaler(h->ws.status, 1.0f, 0, 0, nullptr);
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    if (e != cudaSuccess) {
        cudaFree(h->ws_block);
        delete h;
        return cuda_fail(nullptr, e, "workspace initialisation");
    }
    *out = h;
    return ZERO_OK;
}

int zero_partition_info(zero_handle_t h, uint64_t* psi_pad, uint64_t* shard, uint64_t* offsets,
                        uint64_t* real) {
    if (!h) return fail(nullptr, ZERO_EINVAL, "handle is NULL");
    if (psi_pad) *psi_pad = h->psi_pad;
    if (shard) *shard = h->shard;
    for (int r = 0; r < h->n; ++r) {
        if (offsets) offsets[r] = h->offsets[r];
        if (real) real[r] = h->real[r];
    }
    return ZERO_OK;
}

int zero_set_scaler(zero_handle_t h, float loss_scale, int64_t steps_applied, int32_t state_slot,
                    void* stream) {
    CallRange range_("zero_set_scaler");
    if (!h) return fail(nullptr, ZERO_EINVAL, "handle is NULL");
    if (!std::isfinite(loss_scale) || loss_scale <= 0.0f)
        return fail(h, ZERO_EINVAL, "loss_scale must be finite and > 0");
    if (steps_applied < 0) return fail(h, ZERO_EINVAL, "steps_applied must be >= 0");
    if (state_slot != 0 && !(double_buffered(h) && state_slot == 1))
        return fail(h, ZERO_EINVAL, "state_slot must be 0 (or 1 with a double buffer)");
    h->covered.clear();
    h->rs_calls = 0;
    h->rs_mode = -1;
    cudaError_t e = zg::launch_set_scaler(h->ws.status, loss_scale, steps_applied, state_slot,
                                          static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(h, e, "set_scaler");
    return ZERO_OK;
}

int zero_step(zero_handle_t h, const void* const* grads, void* const* params, float* master, float* m,
              float* v, const zero_hyper_t* hyper, void* stream) {
    CallRange range_("zero_step");
    if (!h) return fail(nullptr, ZERO_EINVAL, "handle is NULL");
    int rc = check_hyper(h, hyper);
    if (rc) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const uint64_t P = h->psi_pad, N = static_cast<uint64_t>(h->n);
    const bool vec8 = (P % 8) == 0;
    const bool any = P > 0;
    zg::Args a = base_args(h, hyper);
    a.base = 0;
    a.count = P;
    a.slot_stride = double_buffered(h) ? P : 0;

    // Bucketed steps (stage 3 always; stage 2 when grads is NULL): the
    // gradients were consumed by the reduce-scatter calls of this step.
    if (h->stage == 3 || (h->stage == 2 && !grads)) {
        const bool st3 = h->stage == 3;
        if (grads) return fail(h, ZERO_EINVAL, "stage 3: grads must be NULL (use zero_reduce_scatter_bucket)");
        if (!params) return fail(h, ZERO_EINVAL, "params is NULL");
        uint64_t covered = 0;
        for (auto& iv : h->covered) covered += iv.second - iv.first;
        if (covered != P)
            return fail(h, ZERO_ESTATE, std::string(st3 ? "stage 3" : "stage 2 (bucketed)") +
                                            ": reduce-scatter buckets cover " + std::to_string(covered) + " of " +
                                            std::to_string(P) + " elements this step");
        int mode = h->rs_mode;
        if (P == 0) {
            rc = resolve_mode(h, hyper, &mode);
            if (rc) return rc;
            if (mode == ZERO_MODE_TWO_PASS_REREAD) mode = ZERO_MODE_TWO_PASS_WS;
        } else if (!same_hyper(*hyper, h->rs_hyper)) {
            return fail(h, ZERO_EINVAL, "zero_step hyper differs from the reduce-scatter calls'");
        }
        const int n_out = st3 ? 1 : h->n;
        if (any) {
            for (int r = 0; r < n_out; ++r) {
                if ((rc = check_ptr(h, params[r], "params[r]"))) return rc;
                a.params[r] = params[r];
            }
            if ((rc = check_ptr(h, master, "master")) || (rc = check_ptr(h, m, "m")) || (rc = check_ptr(h, v, "v")))
                return rc;
        }
        a.master = master;
        a.m = m;
        a.v = v;
        a.bucket_index = h->rs_calls;
        const bool spec = mode == ZERO_MODE_SPECULATIVE;
        if (!spec && any) {
            if ((rc = ensure_ghat(h))) return rc;
            a.ws = h->ws;
        }
        cudaError_t e = zg::launch_finalize3(spec, a, s);
        if (e != cudaSuccess) return cuda_fail(h, e, "finalize");
        if (any) {
            zg::Kind kind = spec ? (st3 ? zg::Kind::kRollbackShard : zg::Kind::kRollbackReplicas)
                                 : (st3 ? zg::Kind::kApplyWsShard : zg::Kind::kApplyWs);
            rc = launch(h, kind, vec8, a, s, spec ? "rollback" : "apply");
            if (rc) return rc;
        }
        h->covered.clear();
        h->rs_calls = 0;
        h->rs_mode = -1;
        if (spec) count(h, 0, 0);
        else count(h, 16 * P, 12 * P + 2 * static_cast<uint64_t>(n_out) * P);
        return ZERO_OK;
    }

    int mode = 0;
    rc = resolve_mode(h, hyper, &mode, /*one_shot=*/h->stage != 0);
    if (rc) return rc;
    if (any) {
        if (!grads) return fail(h, ZERO_EINVAL, "grads is NULL");
        if (!params) return fail(h, ZERO_EINVAL, "params is NULL");
        for (int r = 0; r < h->n; ++r) {
            if ((rc = check_ptr(h, grads[r], "grads[r]"))) return rc;
            if ((rc = check_ptr(h, params[r], "params[r]"))) return rc;
            a.grads[r] = grads[r];
            a.params[r] = params[r];
        }
        if ((rc = check_ptr(h, master, "master")) || (rc = check_ptr(h, m, "m")) || (rc = check_ptr(h, v, "v")))
            return rc;
    }
    a.master = master;
    a.m = m;
    a.v = v;

    if (mode == ZERO_MODE_SPECULATIVE || mode == ZERO_MODE_SPECULATIVE_STAGED) {
        if (mode == ZERO_MODE_SPECULATIVE_STAGED) {
            if (any && pick_vec(vec8, a) != zg::Vec::k8s32)
                return fail(h, ZERO_EINVAL, "staged mode needs 32-byte aligned master/m/v");
            // the bulk copies read the inputs as device global memory only
            const void* ins[zg::kMaxRanks + 3];
            int k = 0;
            for (int r = 0; r < h->n; ++r) ins[k++] = a.grads[r];
            ins[k++] = a.master;
            ins[k++] = a.m;
            ins[k++] = a.v;
            for (int i = 0; i < k; ++i) {
                cudaPointerAttributes pa;
                if (cudaPointerGetAttributes(&pa, ins[i]) != cudaSuccess || pa.type != cudaMemoryTypeDevice) {
                    cudaGetLastError();
                    return fail(h, ZERO_EINVAL, "staged mode reads grads and master/m/v from device memory only");
                }
            }
            zg::Args at = a;
            at.hold_tile1 = h->hold_tile1;
            h->hold_tile1 = 0;
            cudaError_t e = zg::launch_step_tma(h->dtype, at, s);
            if (e != cudaSuccess) return cuda_fail(h, e, "staged step");
        } else if ((rc = launch(h, zg::Kind::kStepSpec, vec8, a, s, "step"))) {
            return rc;
        }
        if ((rc = launch(h, zg::Kind::kFixupReplicas, vec8, a, s, "fixup"))) return rc;
        cudaError_t e = zg::launch_commit_redo(h->ws.status, s);
        if (e != cudaSuccess) return cuda_fail(h, e, "commit");
        count(h, 2 * N * P + 12 * P, 12 * P + 2 * N * P);
        return ZERO_OK;
    }
    if (mode == ZERO_MODE_TWO_PASS_WS) {
        if ((rc = ensure_ghat(h))) return rc;
        a.ws = h->ws;
        if ((rc = launch(h, zg::Kind::kReduceWs, vec8, a, s, "reduce"))) return rc;
        if (h->stage == 0) {
            if ((rc = launch(h, zg::Kind::kApplyStage0, vec8, a, s, "apply"))) return rc;
            count(h, 2 * N * P + 4 * P + 12 * N * P, 4 * P + 12 * N * P + 2 * N * P);
        } else {
            if ((rc = launch(h, zg::Kind::kApplyWs, vec8, a, s, "apply"))) return rc;
            count(h, 2 * N * P + 4 * P + 12 * P, 4 * P + 12 * P + 2 * N * P);
        }
        return ZERO_OK;
    }
    // TWO_PASS_REREAD
    if ((rc = launch(h, zg::Kind::kReduceNoWs, vec8, a, s, "reduce"))) return rc;
    if ((rc = launch(h, zg::Kind::kApplyReread, vec8, a, s, "apply"))) return rc;
    count(h, 4 * N * P + 12 * P, 12 * P + 2 * N * P);
    return ZERO_OK;
}

int zero_gather_bucket(zero_handle_t h, uint64_t a0, uint64_t b0, const void* shard16, void* const* out,
                       void* stream) {
    CallRange range_("zero_gather_bucket");
    if (!h) return fail(nullptr, ZERO_EINVAL, "handle is NULL");
    if (h->stage != 3) return fail(h, ZERO_EINVAL, "zero_gather_bucket is for stage 3");
    if (a0 > b0 || b0 > h->psi_pad) return fail(h, ZERO_EINVAL, "bucket must satisfy 0 <= a <= b <= psi_pad");
    const uint64_t L = b0 - a0, N = static_cast<uint64_t>(h->n);
    if (L == 0) {
        count(h, 0, 0);
        return ZERO_OK;
    }
    int rc = check_ptr(h, shard16, "shard16");
    if (rc) return rc;
    if (!out) return fail(h, ZERO_EINVAL, "out is NULL");
    zg::Args a = base_args(h, nullptr);
    a.grads[0] = shard16;
    for (int r = 0; r < h->n; ++r) {
        if ((rc = check_ptr(h, out[r], "out[r]"))) return rc;
        a.params[r] = out[r];
    }
    a.base = a0;
    a.count = L;
    const bool vec8 = (a0 % 8) == 0 && (L % 8) == 0;
    if ((rc = launch(h, zg::Kind::kGather, vec8, a, static_cast<cudaStream_t>(stream), "gather"))) return rc;
    count(h, 2 * L, 2 * N * L);
    return ZERO_OK;
}

int zero_reduce_scatter_bucket(zero_handle_t h, uint64_t a0, uint64_t b0, const void* const* grads,
                               float* master, float* m, float* v, void* shard16, const zero_hyper_t* hyper,
                               void* stream) {
    CallRange range_("zero_reduce_scatter_bucket");
    if (!h) return fail(nullptr, ZERO_EINVAL, "handle is NULL");
    if (h->stage != 3) return fail(h, ZERO_EINVAL, "zero_reduce_scatter_bucket is for stage 3");
    void* outs[1] = {shard16};
    return rs_bucket(h, a0, b0, grads, master, m, v, outs, hyper, stream);
}

int zero_reduce_scatter_gather_bucket(zero_handle_t h, uint64_t a0, uint64_t b0, const void* const* grads,
                                      float* master, float* m, float* v, void* shard16, const zero_hyper_t* hyper,
                                      uint64_t ga, uint64_t gb, void* const* out, void* stream) {
    CallRange range_("zero_reduce_scatter_gather_bucket");
    if (!h) return fail(nullptr, ZERO_EINVAL, "handle is NULL");
    if (h->stage != 3) return fail(h, ZERO_EINVAL, "zero_reduce_scatter_gather_bucket is for stage 3");
    if (a0 > b0 || b0 > h->psi_pad || ga > gb || gb > h->psi_pad)
        return fail(h, ZERO_EINVAL, "buckets must satisfy 0 <= a <= b <= psi_pad and 0 <= ga <= gb <= psi_pad");
    const uint64_t L = b0 - a0, GL = gb - ga;
    if (L > 0 && GL > 0 && a0 < gb && ga < b0)
        return fail(h, ZERO_EINVAL, "the gathered bucket overlaps the reduce-scattered one");
    int rc = ZERO_OK;
    if (GL > 0) {
        if ((rc = check_ptr(h, shard16, "shard16"))) return rc;
        if (!out) return fail(h, ZERO_EINVAL, "out is NULL");
        for (int r = 0; r < h->n; ++r) {
            if ((rc = check_ptr(h, out[r], "out[r]"))) return rc;
            // both parts may run at once: the outputs must not share memory
            // with what the reduce-scatter reads or writes
            if (overlaps(out[r], 2 * GL, shard16, 2 * h->psi_pad))
                return fail(h, ZERO_EINVAL, "out[r] overlaps the 16-bit shard");
            const uint64_t state_bytes = 4 * h->psi_pad * (double_buffered(h) ? 2 : 1);
            for (const float* st : {master, m, v})
                if (overlaps(out[r], 2 * GL, st, state_bytes))
                    return fail(h, ZERO_EINVAL, "out[r] overlaps master, m or v");
            for (int q = 0; L > 0 && grads && q < h->n; ++q)
                if (overlaps(out[r], 2 * GL, grads[q], 2 * L))
                    return fail(h, ZERO_EINVAL, "out[r] overlaps a gradient row of the reduce-scattered bucket");
        }
    }
    const bool fuse = L > 0 && GL > 0 && bucket_vec8(h, a0, L) && (ga % 8) == 0 && (GL % 8) == 0;
    void* outs[1] = {shard16};
    if (fuse) return rs_bucket(h, a0, b0, grads, master, m, v, outs, hyper, stream, 0, nullptr, ga, GL, out);
    // one part empty, or not 8-wide: the two calls one after the other
    const uint64_t r0 = h->tot_r, w0 = h->tot_w;
    if ((rc = rs_bucket(h, a0, b0, grads, master, m, v, outs, hyper, stream))) return rc;
    if ((rc = zero_gather_bucket(h, ga, gb, shard16, out, stream))) return rc;
    h->last_r = h->tot_r - r0;
    h->last_w = h->tot_w - w0;
    return ZERO_OK;
}

int zero_reduce_scatter_bucket_replicas(zero_handle_t h, uint64_t a0, uint64_t b0, const void* const* grads,
                                        float* master, float* m, float* v, void* const* params,
                                        const zero_hyper_t* hyper, void* stream) {
    CallRange range_("zero_reduce_scatter_bucket_replicas");
    if (!h) return fail(nullptr, ZERO_EINVAL, "handle is NULL");
    if (h->stage != 2) return fail(h, ZERO_EINVAL, "zero_reduce_scatter_bucket_replicas is for stage 2");
    return rs_bucket(h, a0, b0, grads, master, m, v, params, hyper, stream);
}

int zero_quantize_blocks(int dtype, int bits, const void* src16, uint64_t count, void* codes, float* scales,
                         void* stream) {
    CallRange range_("zero_quantize_blocks");
    if (dtype != ZERO_FP16 && dtype != ZERO_BF16) return fail(nullptr, ZERO_EINVAL, "dtype must be fp16 or bf16");
    if (bits != 8 && bits != 4) return fail(nullptr, ZERO_EINVAL, "bits must be 8 or 4");
    if (count == 0) return ZERO_OK;
    if (!src16 || !aligned16(src16)) return fail(nullptr, ZERO_EINVAL, "src16 is NULL or not 16-byte aligned");
    if (!codes || !aligned16(codes)) return fail(nullptr, ZERO_EINVAL, "codes is NULL or not 16-byte aligned");
    if (!scales || !aligned8(scales)) return fail(nullptr, ZERO_EINVAL, "scales is NULL or not 8-byte aligned");
    zg::Args a;
    std::memset(&a, 0, sizeof(a));
    a.grads[0] = src16;
    a.params[0] = codes;
    a.qdst[0] = scales;
    a.count = count;
    a.qbits = bits;
    a.qvec = 1;
    const cudaError_t e = zg::launch_q(zg::QKind::kQuantize, dtype, bits, zg::Vec::k1, a, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(nullptr, e, "quantize");
    return ZERO_OK;
}

int zero_dequantize_blocks(int dtype, int bits, const void* codes, const float* scales, uint64_t count, void* out16,
                           void* stream) {
    CallRange range_("zero_dequantize_blocks");
    if (dtype != ZERO_FP16 && dtype != ZERO_BF16) return fail(nullptr, ZERO_EINVAL, "dtype must be fp16 or bf16");
    if (bits != 8 && bits != 4) return fail(nullptr, ZERO_EINVAL, "bits must be 8 or 4");
    if (count == 0) return ZERO_OK;
    if (!codes || !aligned16(codes)) return fail(nullptr, ZERO_EINVAL, "codes is NULL or not 16-byte aligned");
    if (!scales || !aligned8(scales)) return fail(nullptr, ZERO_EINVAL, "scales is NULL or not 8-byte aligned");
    if (!out16 || !aligned16(out16)) return fail(nullptr, ZERO_EINVAL, "out16 is NULL or not 16-byte aligned");
    zg::Args a;
    std::memset(&a, 0, sizeof(a));
    a.grads[0] = codes;
    a.qsrc[0] = scales;
    a.params[0] = out16;
    a.count = count;
    a.qbits = bits;
    const cudaError_t e = zg::launch_q(zg::QKind::kDequantize, dtype, bits, zg::Vec::k1, a, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(nullptr, e, "dequantize");
    return ZERO_OK;
}

int zero_gather_bucket_q8(zero_handle_t h, uint64_t a0, uint64_t b0, const void* shard16, void* const* codes_out,
                          float* const* scales_out, void* stream) {
    CallRange range_("zero_gather_bucket_q8");
    if (!h) return fail(nullptr, ZERO_EINVAL, "handle is NULL");
    if (h->stage != 3) return fail(h, ZERO_EINVAL, "zero_gather_bucket_q8 is for stage 3");
    if (a0 > b0 || b0 > h->psi_pad) return fail(h, ZERO_EINVAL, "bucket must satisfy 0 <= a <= b <= psi_pad");
    const uint64_t L = b0 - a0, N = static_cast<uint64_t>(h->n);
    if (L == 0) {
        count(h, 0, 0);
        return ZERO_OK;
    }
    int rc = check_ptr(h, shard16, "shard16");
    if (rc) return rc;
    if (!codes_out || !scales_out) return fail(h, ZERO_EINVAL, "codes_out / scales_out is NULL");
    zg::Args a = base_args(h, nullptr);
    a.grads[0] = shard16;
    for (int r = 0; r < h->n; ++r) {
        if ((rc = check_ptr(h, codes_out[r], "codes_out[r]"))) return rc;
        if (!scales_out[r] || !aligned8(scales_out[r])) return fail(h, ZERO_EINVAL, "scales_out[r] is NULL or not 8-byte aligned");
        a.params[r] = codes_out[r];
        a.qdst[r] = scales_out[r];
    }
    a.base = a0;
    a.count = L;
    a.qbits = 8;
    a.qvec = (a0 % 8) == 0 ? 1 : 0;
    a.ctr_slot = next_slot(h);
    const cudaError_t e = zg::launch_q(zg::QKind::kGatherQ8, h->dtype, 8, zg::Vec::k1, a, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(h, e, "quantized gather");
    const uint64_t nb = (L + zg::kQBlock - 1) / zg::kQBlock;
    count(h, 2 * L, N * (L + 8 * nb));
    return ZERO_OK;
}

int zero_reduce_scatter_bucket_q(zero_handle_t h, uint64_t a0, uint64_t b0, int bits, const void* const* codes,
                                 const float* const* scales, float* master, float* m, float* v, void* shard16,
                                 const zero_hyper_t* hyper, void* stream) {
    CallRange range_("zero_reduce_scatter_bucket_q");
    if (!h) return fail(nullptr, ZERO_EINVAL, "handle is NULL");
    if (h->stage != 3) return fail(h, ZERO_EINVAL, "zero_reduce_scatter_bucket_q is for stage 3");
    if (bits != 8 && bits != 4) return fail(h, ZERO_EINVAL, "bits must be 8 or 4");
    void* outs[1] = {shard16};
    return rs_bucket(h, a0, b0, codes, master, m, v, outs, hyper, stream, bits, scales);
}

int zero_get_status(zero_handle_t h, void* stream, zero_result_t* out) {
    CallRange range_("zero_get_status");
    if (!h) return fail(nullptr, ZERO_EINVAL, "handle is NULL");
    if (!out) return fail(h, ZERO_EINVAL, "out is NULL");
    zg::DevStatus st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaMemcpyAsync(&st, h->ws.status, sizeof(st), cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_fail(h, e, "status read");
    out->overflow = st.overflow;
    out->applied = st.applied;
    out->state_slot = st.live_slot;
    out->error = st.error;
    out->grad_norm = st.norm;
    out->clip_coef = st.clip_coef;
    out->loss_scale = st.loss_scale;
    out->reserved = 0.0f;
    out->steps_applied = st.t;
    out->steps_skipped = st.skipped;
    if (st.error) return fail(h, ZERO_ETIMEOUT, "a bounded device wait gave up; the step was skipped");
    return ZERO_OK;
}

int zero_debug_hold_staged(zero_handle_t h, int64_t tile) {
    if (!h) return fail(nullptr, ZERO_EINVAL, "handle is NULL");
    h->hold_tile1 = tile < 0 ? 0 : static_cast<uint64_t>(tile) + 1;
    return ZERO_OK;
}

int zero_set_persistent(zero_handle_t h, uint64_t p0) {
    if (!h) return fail(nullptr, ZERO_EINVAL, "handle is NULL");
    if (h->stage != 3) return fail(h, ZERO_EINVAL, "zero_set_persistent is for stage 3");
    if (p0 > h->psi_pad) return fail(h, ZERO_EINVAL, "p0 must satisfy 0 <= p0 <= psi_pad");
    h->persist_from = p0;
    return ZERO_OK;
}

int zero_bytes_moved(zero_handle_t h, zero_bytes_t* out) {
    if (!h) return fail(nullptr, ZERO_EINVAL, "handle is NULL");
    if (!out) return fail(h, ZERO_EINVAL, "out is NULL");
    const uint64_t P = h->psi_pad, N = static_cast<uint64_t>(h->n);
    out->psi = h->psi;
    out->psi_pad = P;
    out->shard = h->shard;
    out->n_ranks = N;
    out->stage = static_cast<uint64_t>(h->stage);
    // the resident region of a stage-3 handle (zero_set_persistent): each
    // rank keeps its 16-bit copy, which is gathered once per step (after the
    // update) instead of before forward and before backward
    const uint64_t pers = P - h->persist_from;
    switch (h->stage) {
        case 0: out->model_state_bytes_per_rank = 16 * P; break;
        case 1: out->model_state_bytes_per_rank = 4 * P + 12 * P / N; break;
        case 2: out->model_state_bytes_per_rank = 2 * P + 14 * P / N; break;
        default: out->model_state_bytes_per_rank = 16 * P / N + 2 * pers; break;
    }
    if (h->stage == 3) {
        out->comm_elems_paper = 3 * P - pers;
        out->comm_elems_ring = (N - 1) * (3 * P - pers) / N;
    } else {
        out->comm_elems_paper = 2 * P;
        out->comm_elems_ring = 2 * (P / N) * (N - 1);
    }
    out->hbm_read_bytes = h->last_r;
    out->hbm_write_bytes = h->last_w;
    out->hbm_read_total = h->tot_r;
    out->hbm_write_total = h->tot_w;
    return ZERO_OK;
}

const char* zero_last_error(zero_handle_t h) {
    if (!h) return g_init_error.c_str();
    return h->err.c_str();
}

void zero_destroy(zero_handle_t h) {
    if (!h) return;
    int prev = 0;
    cudaGetDevice(&prev);
    cudaSetDevice(h->device);
    cudaDeviceSynchronize();
    if (h->ws.ghat) cudaFree(h->ws.ghat);
    if (h->ws_block) cudaFree(h->ws_block);
    cudaSetDevice(prev);
    delete h;
}

}  // extern "C"
