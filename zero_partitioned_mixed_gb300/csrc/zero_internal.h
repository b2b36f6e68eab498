// Internal types shared by the host C ABI (zero_api.cpp) and the kernels
// (zero_kernels.cu).  Not part of the public interface.
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda_runtime.h>

namespace zg {

constexpr int kMaxRanks = 64;
constexpr int kMaxBlocks = 4096;    // per-block norm partials of one launch
constexpr int kMaxBuckets = 4096;   // reduce-scatter calls of one ZeRO-3 step
constexpr int kThreads = 256;

// Dynamic chunk scheduling (zero_device.cuh): a launch's CTAs take chunks of
// kChunkU * kThreads vectors from a counter; norm partials are formed per
// chunk and summed per group of kGroup chunks, so they do not depend on
// which CTA took which chunk.
constexpr int kChunkU = 4;
constexpr uint64_t kChunkVec = static_cast<uint64_t>(kChunkU) * kThreads;
constexpr int kGroup = 32;
constexpr uint64_t kDirectChunks = 4096;   // up to this many chunks, no group stage
constexpr int kCtrSlots = 64;       // launches of one handle that may be in flight at once

// Vectors per thread in a chunk: UMAX for large launches, fewer (down to 1)
// for smaller ones, so that a launch has about TARGET chunks or more --
// enough for every CTA of the persistent grid and a short tail.  A function
// of the launch's size only, so the chunk partials stay deterministic.
// UMAX is the kernel's own cap and TARGET the chunk count it aims at (a
// launch gets about TARGET chunks or more, unless UMAX caps U first).
// Measured per kernel: the stage 1/2 step does best with UMAX 16 and TARGET
// 16384 (long chunks for large launches, many for mid-sized ones), the
// two-pass kernels with TARGET 16384, the reduce-scatter into replicas with
// 8192, the gather with the default, the reduce-scatter into the shard with
// the default (4096 at N <= 2).
// Any (UMAX, TARGET) keeps the partials deterministic.
constexpr uint64_t kMinChunks = 2048;        // the default TARGET
constexpr uint64_t kMaxChunkTarget = 16384;  // the largest TARGET of a kernel that writes chunk partials
__host__ __device__ inline int chunk_u(uint64_t nvec, int umax, uint64_t target = kMinChunks) {
    const uint64_t u = nvec / (static_cast<uint64_t>(kThreads) * target);
    return u >= static_cast<uint64_t>(umax) ? umax : (u < 1 ? 1 : static_cast<int>(u));
}
__host__ __device__ inline uint64_t chunk_len(uint64_t nvec, int umax, uint64_t target = kMinChunks) {
    return static_cast<uint64_t>(chunk_u(nvec, umax, target)) * kThreads;
}
__host__ __device__ inline uint64_t chunk_total(uint64_t nvec, int umax, uint64_t target = kMinChunks) {
    const uint64_t len = chunk_len(nvec, umax, target);
    return (nvec + len - 1) / len;
}
template <int UMAX = kChunkU, uint64_t TARGET = kMinChunks>
__host__ __device__ inline int chunk_u(uint64_t nvec) { return chunk_u(nvec, UMAX, TARGET); }
template <int UMAX = kChunkU, uint64_t TARGET = kMinChunks>
__host__ __device__ inline uint64_t chunk_len(uint64_t nvec) { return chunk_len(nvec, UMAX, TARGET); }
template <int UMAX = kChunkU, uint64_t TARGET = kMinChunks>
__host__ __device__ inline uint64_t chunk_total(uint64_t nvec) { return chunk_total(nvec, UMAX, TARGET); }

// Chunks and groups of any launch over at most `elems` elements (worst case:
// 1-wide vectors at kChunkU vectors per thread; below that a launch has at
// most 2 * TARGET chunks).
inline uint64_t max_chunks(uint64_t elems) {
    const uint64_t a = elems / kChunkVec + 1, b = 2 * kMaxChunkTarget + 1;
    return a > b ? a : b;
}
inline uint64_t max_groups(uint64_t elems) { return max_chunks(elems) / kGroup + 1; }

enum Dtype : int { kFp16 = 0, kBf16 = 1 };

// Adam coefficients of one step, each rounded once to fp32 from double.
struct StepScalars {
    float b1, b2, a1, a2, eps, dfac, step_size, bc2s;
};

struct HyperDev {
    float lr, beta1, beta2, eps, weight_decay, max_norm;
};

// Device-resident state of a handle.  Written only by the last block of a
// step's reducing kernel (or by the one-block finaliser), read by the next
// kernels on the stream.
struct DevStatus {
    float loss_scale;
    int32_t live_slot;
    int64_t t;          // applied steps
    int64_t skipped;
    int32_t overflow;
    int32_t applied;
    double norm;
    double clip_coef;   // fp32 factor applied, as double (1.0 when none)
    float clip_f;
    int32_t use_clip;
    int32_t error;
    int32_t redo;       // speculative step whose norm needs clipping: redo it from the old slot
    StepScalars sc;     // coefficients of the step being applied (two-pass)
    uint32_t ticket;    // last-block counter; returns to 0 after every launch
    uint32_t stop;      // one-pass step: a non-finite gradient was seen, the pass may stop
                        // (the step is skipped); returns to 0 when the pass finalises
    uint64_t hwm1;      // one-pass step: 1 + a bound on the vectors it wrote (every write is
                        // below it); 0 = unknown (the whole range).  Reset after each step.
    // The scalars of step sc_t under the hyper-parameters sc_key, computed once
    // by the thread that finalised the bucketed step before (sc_t = its t + 1).
    // A one-pass kernel whose t + 1 and hyper-parameters match reads them
    // instead of computing them in every CTA; a step of one launch computes
    // its own (the cost only moves between kernels there).
    StepScalars sc_next;
    HyperDev sc_key;
    int64_t sc_t;
};

// Per-launch chunk counter: grabs made so far; zero between launches (the
// CTA that makes a launch's last grab resets it).
struct ChunkCtr {
    unsigned long long next;
    unsigned long long pad;
};

struct Workspace {
    DevStatus* status;
    double* partials;      // [kMaxBlocks]
    int32_t* flags;        // [kMaxBlocks]
    double* bucket_norm;   // [kMaxBuckets]
    int32_t* bucket_flag;  // [kMaxBuckets]
    float* ghat;           // [psi_pad] fp32 averaged gradient, or null
    ChunkCtr* ctrs;        // [kCtrSlots], zero between launches
    double* chunk_part;    // [max_chunks(psi_pad)] norm partial of each chunk
    double* group_part;    // [max_groups(psi_pad)] norm partial of each group of chunks
    uint32_t* group_ticket;  // [max_groups(psi_pad)], zero between launches
};

// Everything a launch needs, passed by value as a __grid_constant__ param.
struct Args {
    const void* grads[kMaxRanks];  // N rank buffers (16-bit)
    void* params[kMaxRanks];       // N replicas, or [0] = 16-bit shard
    int n_ranks;
    int stage;
    uint64_t psi;        // real elements; global indices >= psi are padding
    uint64_t psi_pad;
    uint64_t base;       // global index of the launch's first element
    uint64_t count;      // elements processed by the launch
    float* master;       // slot 0 (or replica 0 for stage 0)
    float* m;
    float* v;
    uint64_t slot_stride;  // floats between state slots (double buffer), else 0
    HyperDev hyper;
    Workspace ws;
    int bucket_index;
    // ZeRO++ block-quantized exchange (zero_quant.cu)
    const float* qsrc[kMaxRanks];  // per-rank {scale, lo} pairs of quantized inputs
    float* qdst[kMaxRanks];        // per-rank {scale, lo} pairs of quantized outputs
    int qbits;                     // 8 or 4
    int qvec;                      // 1: 16-bit source 16-byte aligned at every block start
    // staged step (zero_tma.cu): 1 + the tile at which CTA 0 stops issuing
    // its copies, so that its bounded waits run out (0: never)
    uint64_t hold_tile1;
    int ctr_slot;          // chunked launches: this launch's counter, ws.ctrs[ctr_slot]
    // reduce-scatter fused with the gather of another bucket
    // (zero_reduce_scatter_gather_bucket): after the reduce-scatter's chunks the
    // launch copies params[0][gbase, gbase + gcount) to every gout[r]
    void* gout[kMaxRanks];
    uint64_t gbase;
    uint64_t gcount;
};

enum class Kind : int {
    kStepSpec,        // stages 1/2: one pass, shadow slot
    kReduceWs,        // two-pass pass 1, writes g_hat to workspace
    kReduceNoWs,      // two-pass pass 1, norm/flag only
    kApplyWs,         // two-pass pass 2 from workspace -> replicas
    kApplyReread,     // two-pass pass 2 re-reducing grads -> replicas
    kApplyWsShard,    // stage 3 two-pass pass 2 -> 16-bit shard
    kApplyStage0,     // stage 0 pass 2: N state replicas
    kRollbackReplicas,
    kRollbackShard,
    kFixupReplicas,   // after kStepSpec: roll back on overflow, or redo with clipping
    kGather,
    kRsSpec,          // stage 3 bucket reduce-scatter + fused speculative Adam
    kRsWs,            // bucket reduce-scatter into the workspace (stages 2/3)
    kRsSpecReplicas,  // stage 2 bucket reduce-scatter + fused speculative Adam + all-gather
    kRsSpecGather,    // kRsSpec, then the gather of another bucket in the same launch (8-wide only)
    kRsWsGather,      // kRsWs, then the gather of another bucket in the same launch (8-wide only)
};

// Per-thread vector width of a launch: 8 elements with 256-bit fp32 accesses
// (state and g_hat 32-byte aligned), 8 elements with 128-bit fp32 accesses,
// or one element.
enum class Vec : int { k8s32, k8s16, k1 };

// Launchers (zero_kernels.cu).  Return the cudaError_t of the launch.
cudaError_t launch(Kind kind, int dtype, Vec vec, const Args& a, cudaStream_t s, int* grid_out);
cudaError_t launch_finalize3(bool spec, const Args& a, cudaStream_t s);
cudaError_t launch_set_scaler(DevStatus* st, float loss_scale, int64_t t, int32_t slot, cudaStream_t s);
cudaError_t launch_commit_redo(DevStatus* st, cudaStream_t s);

// The stage 1/2 speculative step with bulk-copy staging (zero_tma.cu), and
// its pipeline depth for N ranks (0: not available for that N).
cudaError_t launch_step_tma(int dtype, const Args& a, cudaStream_t s);
int tma_stages(int n_ranks);

constexpr int kQBlock = 256;   // ZeRO++ quantization block (elements)

enum class QKind : int {
    kQuantize,     // one 16-bit buffer -> codes + {scale, lo}
    kDequantize,   // codes + {scale, lo} -> one 16-bit buffer
    kGatherQ8,     // ZeRO-3 gather: shard bucket -> N copies of int8 codes + scales
    kRsQSpec,      // ZeRO-3 reduce-scatter of N quantized gradients + fused speculative AdamW
    kRsQWs,        // ZeRO-3 reduce-scatter of N quantized gradients into the workspace
};

// Launcher of the ZeRO++ kernels (zero_quant.cu).
cudaError_t launch_q(QKind kind, int dtype, int bits, Vec vec, const Args& a, cudaStream_t s);

// Message returned by zero_last_error(NULL) for calls that take no handle.
void set_global_error(const char* msg);

}  // namespace zg
