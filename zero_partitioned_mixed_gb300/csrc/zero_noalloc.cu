// zero_step_noalloc: the two-pass ZeRO step (stages 1/2) for callers that
// cannot allocate device memory.
//
// Who needs it: code that runs where cudaMalloc is not allowed or not
// wanted -- inside a framework whose caching allocator owns the device
// memory and must not see a foreign cudaMalloc (which also synchronises the
// whole device), or under a fixed memory budget decided before training
// starts.  zero_init_partition allocates a workspace, so such callers
// cannot use the handle-based entry points.
//
// Instead, every piece of scratch this path needs -- the status word, the
// norm partials and flags, the chunk counters, and the fp32 averaged gradient of up to
// kNoAllocMaxPsiPad elements -- lives in one file-scope __device__ array.
// Each GPU that loads the library holds that array until the process exits.
// The kernels are the library's existing two-pass kernels; only the place
// their scratch lives differs.
//
// The loss scale and the step count t are host arguments: a caller passes
// the values that the previous call's result reported, so it reads that
// result back (after synchronising the stream) before the next call.

#include <cstdint>
#include <cstring>
#include <mutex>
#include <string>

#include <cuda_runtime.h>

#include "zero_gb300.h"
#include "zero_internal.h"

namespace {

constexpr uint64_t kNoAllocMaxPsiPad = ZERO_NOALLOC_MAX_PSI_PAD;
constexpr size_t kStatusBytes = 256;
constexpr size_t kPartialBytes = static_cast<size_t>(zg::kMaxBlocks) * sizeof(double);
constexpr size_t kFlagBytes = static_cast<size_t>(zg::kMaxBlocks) * sizeof(int32_t);
constexpr size_t kGhatBytes = static_cast<size_t>(kNoAllocMaxPsiPad) * sizeof(float);
constexpr size_t round32(size_t x) { return (x + 31) / 32 * 32; }
// chunk scheduling: counters and group tickets (zeroed every call), chunk and group partials
constexpr size_t kCtrBytes = round32(static_cast<size_t>(zg::kCtrSlots) * sizeof(zg::ChunkCtr));
constexpr size_t kChunks = kNoAllocMaxPsiPad / zg::kChunkVec + 1 > 2 * zg::kMaxChunkTarget + 1
                               ? kNoAllocMaxPsiPad / zg::kChunkVec + 1
                               : 2 * zg::kMaxChunkTarget + 1;
constexpr size_t kGroups = kChunks / zg::kGroup + 1;
constexpr size_t kTicketBytes = round32(kGroups * sizeof(uint32_t));
constexpr size_t kChunkPartBytes = round32(kChunks * sizeof(double));
constexpr size_t kGroupPartBytes = round32(kGroups * sizeof(double));
constexpr size_t kScratchBytes = kStatusBytes + kPartialBytes + kFlagBytes + kGhatBytes + kCtrBytes + kTicketBytes +
                                 kChunkPartBytes + kGroupPartBytes;
static_assert(sizeof(zg::DevStatus) <= kStatusBytes, "status must fit its slot");
static_assert(kStatusBytes % 32 == 0 && kPartialBytes % 32 == 0 && kFlagBytes % 32 == 0 && kGhatBytes % 32 == 0,
              "scratch regions stay 32-byte aligned");

// The scratch.  Host code must not pass &g_noalloc_scratch to a kernel: on
// the host that name is a stand-in, not a device address.  Its device
// address comes from cudaGetSymbolAddress, once per device.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
unsigned char* g_scratch_ptr[kMaxDevices] = {};

int fail(int code, const std::string& msg) {
    zg::set_global_error(msg.c_str());
    return code;
}

// Device address of the scratch on the current device (set up on first use).
int scratch_address(int dev, unsigned char** out) {
    if (dev < 0 || dev >= kMaxDevices) return fail(ZERO_EINVAL, "device index out of range");
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_scratch_ptr[dev]) {
        void* p = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess || !p)
            return fail(ZERO_ECUDA, std::string("cudaGetSymbolAddress of the static scratch: ") +
                                        cudaGetErrorString(e));
        g_scratch_ptr[dev] = static_cast<unsigned char*>(p);
    }
    *out = g_scratch_ptr[dev];
    return ZERO_OK;
}

__global__ void k_export_result(const zg::DevStatus* st, zero_result_t* out) {
    out->overflow = st->overflow;
    out->applied = st->applied;
    out->state_slot = 0;
    out->error = st->error;
    out->grad_norm = st->norm;
    out->clip_coef = st->clip_coef;
    out->loss_scale = st->loss_scale;
    out->reserved = 0.0f;
    out->steps_applied = st->t;
    out->steps_skipped = st->skipped;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" uint64_t zero_noalloc_scratch_bytes(void) { return kScratchBytes; }

extern "C" int zero_step_noalloc(uint64_t psi, int n_ranks, int stage, int dtype, int align,
                                 const void* const* grads, void* const* params, float* master, float* m,
                                 float* v, const zero_hyper_t* hyper, float loss_scale, int64_t steps_applied,
                                 zero_result_t* result, void* stream) {
    if (n_ranks < 1 || n_ranks > ZERO_MAX_RANKS) return fail(ZERO_EINVAL, "n_ranks must be in 1..64");
    if (stage != 1 && stage != 2) return fail(ZERO_EINVAL, "zero_step_noalloc runs stages 1 and 2");
    if (dtype != ZERO_FP16 && dtype != ZERO_BF16) return fail(ZERO_EINVAL, "dtype must be fp16 or bf16");
    if (align < 1) return fail(ZERO_EINVAL, "align must be >= 1");
    if (!hyper) return fail(ZERO_EINVAL, "hyper is NULL");
    if (hyper->mode != ZERO_MODE_AUTO && hyper->mode != ZERO_MODE_TWO_PASS_WS)
        return fail(ZERO_EINVAL, "zero_step_noalloc is two-pass: mode must be AUTO or TWO_PASS_WS");
    const float hv[] = {hyper->lr, hyper->beta1, hyper->beta2, hyper->eps, hyper->weight_decay, hyper->max_norm};
    for (float x : hv)
        if (!(x == x) || x > 3.0e38f || x < -3.0e38f) return fail(ZERO_EINVAL, "hyper-parameters must be finite");
    if (!(hyper->beta1 >= 0.0f && hyper->beta1 < 1.0f && hyper->beta2 >= 0.0f && hyper->beta2 < 1.0f))
        return fail(ZERO_EINVAL, "beta1 and beta2 must lie in [0, 1)");
    if (!(loss_scale > 0.0f && loss_scale <= 3.0e38f)) return fail(ZERO_EINVAL, "loss_scale must be finite and > 0");
    if (steps_applied < 0) return fail(ZERO_EINVAL, "steps_applied must be >= 0");
    const uint64_t unit = static_cast<uint64_t>(n_ranks) * static_cast<uint64_t>(align);
    if (psi > kNoAllocMaxPsiPad) {
        return fail(ZERO_EINVAL, "psi " + std::to_string(psi) + " exceeds the static scratch of zero_step_noalloc (" +
                                     std::to_string(kNoAllocMaxPsiPad) + " elements); use zero_step");
    }
    const uint64_t P = (psi + unit - 1) / unit * unit;
    if (P > kNoAllocMaxPsiPad) {
        return fail(ZERO_EINVAL, "psi_pad " + std::to_string(P) + " exceeds the static scratch of zero_step_noalloc (" +
                                     std::to_string(kNoAllocMaxPsiPad) + " elements); use zero_step");
    }
    if (!result || (reinterpret_cast<uintptr_t>(result) & 7u)) return fail(ZERO_EINVAL, "result must be an 8-byte aligned device pointer");
    {
        // the result is written by a kernel: refuse memory the GPU cannot
        // reach (pageable host memory) before anything is launched
        cudaPointerAttributes pa;
        const cudaError_t pe = cudaPointerGetAttributes(&pa, result);
        if (pe != cudaSuccess || (pa.type != cudaMemoryTypeDevice && pa.type != cudaMemoryTypeManaged &&
                                  pa.type != cudaMemoryTypeHost)) {
            cudaGetLastError();
            return fail(ZERO_EINVAL, "result must be device, managed or pinned host memory");
        }
    }

    zg::Args a;
    std::memset(&a, 0, sizeof(a));
    if (P > 0) {
        if (!grads || !params) return fail(ZERO_EINVAL, "grads and params must not be NULL");
        for (int r = 0; r < n_ranks; ++r) {
            if (!grads[r] || !aligned16(grads[r])) return fail(ZERO_EINVAL, "grads[r] is NULL or not 16-byte aligned");
            if (!params[r] || !aligned16(params[r])) return fail(ZERO_EINVAL, "params[r] is NULL or not 16-byte aligned");
            a.grads[r] = grads[r];
            a.params[r] = params[r];
        }
        if (!master || !m || !v || !aligned16(master) || !aligned16(m) || !aligned16(v))
            return fail(ZERO_EINVAL, "master, m and v must be 16-byte aligned device pointers");
    }

    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail(ZERO_ECUDA, std::string("cudaGetDevice: ") + cudaGetErrorString(e));
    unsigned char* base = nullptr;
    int rc = scratch_address(dev, &base);
    if (rc) return rc;

    a.n_ranks = n_ranks;
    a.stage = stage;
    a.psi = psi;
    a.psi_pad = P;
    a.base = 0;
    a.count = P;
    a.master = master;
    a.m = m;
    a.v = v;
    a.slot_stride = 0;
    a.hyper.lr = hyper->lr;
    a.hyper.beta1 = hyper->beta1;
    a.hyper.beta2 = hyper->beta2;
    a.hyper.eps = hyper->eps;
    a.hyper.weight_decay = hyper->weight_decay;
    a.hyper.max_norm = hyper->max_norm;
    a.ws.status = reinterpret_cast<zg::DevStatus*>(base);
    a.ws.partials = reinterpret_cast<double*>(base + kStatusBytes);
    a.ws.flags = reinterpret_cast<int32_t*>(base + kStatusBytes + kPartialBytes);
    a.ws.bucket_norm = nullptr;
    a.ws.bucket_flag = nullptr;
    a.ws.ghat = reinterpret_cast<float*>(base + kStatusBytes + kPartialBytes + kFlagBytes);
    unsigned char* sched = base + kStatusBytes + kPartialBytes + kFlagBytes + kGhatBytes;
    a.ws.ctrs = reinterpret_cast<zg::ChunkCtr*>(sched);
    a.ws.group_ticket = reinterpret_cast<uint32_t*>(sched + kCtrBytes);
    a.ws.chunk_part = reinterpret_cast<double*>(sched + kCtrBytes + kTicketBytes);
    a.ws.group_part = reinterpret_cast<double*>(sched + kCtrBytes + kTicketBytes + kChunkPartBytes);

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // 8-wide with 256-bit fp32 accesses when the caller's state is 32-byte
    // aligned (the scratch's g_hat region is); 128-bit otherwise
    const bool s32 = ((reinterpret_cast<uintptr_t>(master) | reinterpret_cast<uintptr_t>(m) |
                       reinterpret_cast<uintptr_t>(v)) & 31u) == 0;
    const zg::Vec vec = (P % 8) != 0 ? zg::Vec::k1 : (s32 ? zg::Vec::k8s32 : zg::Vec::k8s16);
    // the status word (and its last-block ticket) must start from zero
    e = cudaMemsetAsync(a.ws.status, 0, kStatusBytes, s);
    // and the chunk counters and group tickets
    if (e == cudaSuccess) e = cudaMemsetAsync(sched, 0, kCtrBytes + kTicketBytes, s);
    if (e == cudaSuccess) e = zg::launch_set_scaler(a.ws.status, loss_scale, steps_applied, 0, s);
    a.ctr_slot = 0;
    if (e == cudaSuccess) e = zg::launch(zg::Kind::kReduceWs, dtype, vec, a, s, nullptr);
    a.ctr_slot = 1;
    if (e == cudaSuccess) e = zg::launch(zg::Kind::kApplyWs, dtype, vec, a, s, nullptr);
    if (e == cudaSuccess) {
        k_export_result<<<1, 1, 0, s>>>(a.ws.status, result);
        e = cudaGetLastError();
    }
    if (e != cudaSuccess) return fail(ZERO_ECUDA, std::string("zero_step_noalloc launch: ") + cudaGetErrorString(e));
    return ZERO_OK;
}
