// Kernels of the partitioned mixed-precision ZeRO step, written for sm_103a.
//
// The N simulated ranks of the method live in one GPU's HBM, so each
// collective becomes an HBM stream fused into an update kernel:
//   reduce-scatter  -> every thread reads the N ranks' 16-bit gradients of
//                      its 8 elements and sums them in rank order in fp32;
//   scalar all-reduce of the norm and overflow flag -> partials per chunk
//                      of work (and per group of chunks) that the last
//                      block to finish sums in a fixed order (a ticket
//                      counter, no spinning);
//   all-gather / broadcast -> the thread writes the RNE-cast 16-bit result
//                      to all N replicas.
// Every kernel is an HBM-bound stream: 128-bit (16-bit data) and 256-bit
// (fp32 data) loads and stores of contiguous 8-element groups, on a
// persistent grid sized from the SM count and the kernel's occupancy whose
// CTAs take chunks of work from a counter (zero_device.cuh).  There is no contraction,
// so no tensor-core path.
//
// Arithmetic follows the method exactly as the CPU oracle states it: fp32
// operations each rounded once (explicit _rn intrinsics, built with
// -fmad=false), ranks summed from +0 in order 0..N-1, IEEE divide and
// square root, round-to-nearest-even casts.  Sources, by page and section:
// "ZeRO: Memory Optimizations Toward Training Trillion Parameter Models"
// (summary) Sec. 3.1, Sec. 5, Sec. 7 and the residual-state discussion of
// the flattened gradient-norm buffer; "CMU 11-868 L18" ZeRO-1/2/3 call
// sequences; "zero-stages-simulation" README partition and schedule.

#include "zero_device.cuh"

namespace zg {
namespace {

// ------------------------------------------------------------------ kernels
// The one-pass step's cap on vectors per thread in a chunk: fewer chunk
// barriers for its long iterations (ψ = 2^29, N = 2: 2.67 against 2.77 ms
// at 4; the flat 1.5e9 step: 12.45 against 12.54 ms).
constexpr int kStepChunkU = 16;
// Chunk targets (chunks a launch aims at before the cap): a mid-sized launch
// is cut finer so that its last chunks end together.  GPT-2 small (1.2e8
// parameters, N = 8): the one-pass step 1.048 ms at 16384 against 1.087 ms
// at 2048, the two-pass step 1.203 against 1.213 ms; ZeRO-2 buckets of 5e7
// reduced into the replicas 13.07 ms at 8192 against 13.21 ms at 2048.  The
// flat 1.5e9 step is capped first and does not change.
constexpr uint64_t kStepChunks = 16384;
constexpr uint64_t kTwoPassChunks = 16384;
constexpr uint64_t kRsReplicaChunks = 8192;
constexpr uint64_t kRsSmallNChunks = 4096;
static_assert(kStepChunks <= kMaxChunkTarget && kTwoPassChunks <= kMaxChunkTarget &&
                  kRsReplicaChunks <= kMaxChunkTarget && kRsSmallNChunks <= kMaxChunkTarget,
              "the workspace holds the partials of at most 2 * kMaxChunkTarget chunks");
// The step's target is kStepChunks from N = 8 up.  With N <= 4 an iteration
// moves few bytes, the chunk bookkeeping weighs more, and the default target
// measured better (the bandwidth sweep's stage-1 points at N = 2: 2^24
// 0.119 against 0.129 ms, 2^27 0.696 against 0.716 ms).
__host__ __device__ inline uint64_t step_chunk_target(int n_ranks) { return n_ranks <= 4 ? kMinChunks : kStepChunks; }
// Stages 1/2, one pass: reduce-scatter + unscale + flag + norm partial +
// AdamW from the live slot into the shadow slot + cast + all-gather.  The
// last block commits the shadow slot, or records the overflow (the
// rollback kernel then restores the replicas).
// MINB CTAs per SM: 3 (80 registers), or 4 (64 registers, some spill) for
// N <= 2, where an iteration moves few bytes and the extra warps keep more
// loads in flight: psi = 2^29, N = 2: 2.60 against 2.70 ms; at N = 4 and 8
// the fourth CTA was slower (3.25 against 3.21 ms, 4.54 against 4.46 ms).
constexpr int kSmallN = 2;
template <int DT, class IO, int MINB>
__global__ void __launch_bounds__(kThreads, MINB) k_step_spec(const __grid_constant__ Args a) {
    pdl_enter();
    constexpr int W = IO::W;
    __shared__ Pro pro;
    __shared__ unsigned long long s_c[2];
    __shared__ double s_wp[2][kThreads / 32];
    prologue_reduce(a, pro, true);
    const uint64_t src = static_cast<uint64_t>(pro.live) * a.slot_stride;
    const uint64_t dst = static_cast<uint64_t>(pro.live ^ 1) * a.slot_stride;
    const uint64_t nvec = a.count / W;
    const uint64_t target = step_chunk_target(a.n_ranks);
    const uint64_t clen = chunk_len(nvec, kStepChunkU, target);
    const uint64_t nchunks = chunk_total(nvec, kStepChunkU, target);
    const int U = chunk_u(nvec, kStepChunkU, target);
    ChunkCtr* ctr = a.ws.ctrs + a.ctr_slot;
    int bad = 0;
    // Overflow is the existence of one non-finite averaged gradient, and an
    // overflowed step changes no state (the fixup kernel restores the
    // replicas from the old master).  So the thread that finds one raises
    // `stop`, and the CTAs leave at the end of their chunk; the flag is read
    // one vector ahead, off the critical path.
    volatile uint32_t* stop = &a.ws.status->stop;
    uint32_t seen = 0;
    uint64_t reach = 0;   // thread 0: 1 + the last chunk this CTA worked on
    Chunks ch(ctr, s_c, nchunks);
    for (;;) {
        const uint64_t c = ch.current();
        if (c >= nchunks) break;
        ch.prefetch();
        reach = c + 1;
        double cacc = 0.0;
        for (int u = 0; u < U; ++u) {
            const uint64_t vi = chunk_vec(c, clen, u);
            if (vi >= nvec) break;
            const uint32_t seen_next = *stop;
            const uint64_t gi = vi * W;
            float g[W], p[W], m[W], v[W];
            reduce_group<DT, IO>(a, gi, pro, g);
            IO::ldf(a.master + src, gi, p);
            IO::ldf(a.m + src, gi, m);
            IO::ldf(a.v + src, gi, v);
            const int valid = valid_count(gi, W, a.psi);
            norm_group<W>(g, valid, cacc, bad);
            if (bad) {
                *stop = 1u;
                break;
            }
            seen = seen_next;
            uint32_t q[W];
#pragma unroll
            for (int k = 0; k < W; ++k) {
                if (k < valid) {
                    adam1(g[k], p[k], m[k], v[k], pro.sc);
                } else {
                    p[k] = 0.0f; m[k] = 0.0f; v[k] = 0.0f;
                }
                q[k] = narrow<DT>(p[k]);
            }
            IO::stf(a.master + dst, gi, p);
            IO::stf(a.m + dst, gi, m);
            IO::stf(a.v + dst, gi, v);
            for (int r = 0; r < a.n_ranks; ++r) IO::st16(a.params[r], gi, q);
        }
        const int leave = close_chunk(a.ws, c, nchunks, cacc, s_wp, ch.parity(), static_cast<int>(seen) | bad);
        ch.advance();
        if (leave) break;
    }
    // a CTA works on its chunks in increasing order: every vector written
    // lies below the largest reach, which bounds an overflow rollback
    if (threadIdx.x == 0) atomicMax(reinterpret_cast<unsigned long long*>(&a.ws.status->hwm1), reach * clen + 1ull);
    const int flag = __syncthreads_or(bad);
    if (publish(a, 0.0, flag, a.ws.partials, a.ws.flags)) {
        double q;
        int f;
        gather_groups(a.ws, nchunks, gridDim.x, q, f);
        if (f) reset_groups(a.ws, nchunks);
        if (threadIdx.x == 0) {
            DevStatus* st = a.ws.status;
            ctr->next = 0ull;   // a pass cut short made fewer than nchunks grabs
            if (f) status_skip(st, q);
            else status_decide_spec(st, q, a.hyper);
            st->stop = 0u;
            st->ticket = 0u;
        }
    }
}

// Two-pass, pass 1: reduce + unscale + flag + norm partial (+ fp32 g_hat to
// the workspace).  The last block decides: skip, or clip factor and step
// scalars for pass 2.
template <int DT, class IO, bool WS>
__global__ void __launch_bounds__(kThreads) k_reduce(const __grid_constant__ Args a) {
    pdl_enter();
    constexpr int W = IO::W;
    __shared__ Pro pro;
    __shared__ unsigned long long s_c[2];
    __shared__ double s_wp[2][kThreads / 32];
    prologue_reduce(a, pro, false);
    const uint64_t nvec = a.count / W;
    const uint64_t clen = chunk_len<kChunkU, kTwoPassChunks>(nvec);
    const uint64_t nchunks = chunk_total<kChunkU, kTwoPassChunks>(nvec);
    const int U = chunk_u<kChunkU, kTwoPassChunks>(nvec);
    ChunkCtr* ctr = a.ws.ctrs + a.ctr_slot;
    int bad = 0;
    Chunks ch(ctr, s_c, nchunks);
    for (;;) {
        const uint64_t c = ch.current();
        if (c >= nchunks) break;
        ch.prefetch();
        double cacc = 0.0;
        for (int u = 0; u < U; ++u) {
            const uint64_t vi = chunk_vec(c, clen, u);
            if (vi >= nvec) break;
            const uint64_t gi = vi * W;
            float g[W];
            reduce_group<DT, IO>(a, gi, pro, g);
            const int valid = valid_count(gi, W, a.psi);
            norm_group<W>(g, valid, cacc, bad);
            if (WS) {
#pragma unroll
                for (int k = 0; k < W; ++k)
                    if (k >= valid) g[k] = 0.0f;
                IO::stf(a.ws.ghat, gi, g);
            }
        }
        close_chunk(a.ws, c, nchunks, cacc, s_wp, ch.parity(), 0);
        ch.advance();
    }
    const int flag = __syncthreads_or(bad);
    if (publish(a, 0.0, flag, a.ws.partials, a.ws.flags)) {
        double q;
        int f;
        gather_groups(a.ws, nchunks, gridDim.x, q, f);
        if (threadIdx.x == 0) {
            ctr->next = 0ull;
            DevStatus* st = a.ws.status;
            if (f) status_skip(st, q);
            else status_decide_two_pass(st, q, a.hyper);
            st->ticket = 0u;
        }
    }
}

// Two-pass, pass 2 (stages 1/2/3): skip on overflow; else AdamW in place on
// the live slot with g_hat from the workspace (SRC_WS) or re-reduced from
// the N gradients, clipped if decided, then the 16-bit result to the N
// replicas (stages 1/2) or to the shard (stage 3, TO_SHARD).
template <int DT, class IO, bool SRC_WS, bool TO_SHARD>
__global__ void __launch_bounds__(kThreads) k_apply(const __grid_constant__ Args a) {
    pdl_enter();
    constexpr int W = IO::W;
    __shared__ Pro pro;
    __shared__ unsigned long long s_c[2];
    prologue_reduce(a, pro, false);
    if (pro.overflow) return;   // every CTA: the counter stays untouched
    const uint64_t off = static_cast<uint64_t>(pro.live) * a.slot_stride;
    const uint64_t nvec = a.count / W;
    const uint64_t clen = chunk_len<kChunkU, kTwoPassChunks>(nvec);
    const uint64_t nchunks = chunk_total<kChunkU, kTwoPassChunks>(nvec);
    const int U = chunk_u<kChunkU, kTwoPassChunks>(nvec);
    ChunkCtr* ctr = a.ws.ctrs + a.ctr_slot;
    Chunks ch(ctr, s_c, nchunks);
    for (;;) {
      const uint64_t c = ch.current();
      if (c >= nchunks) break;
      ch.prefetch();
      for (int u = 0; u < U; ++u) {
        const uint64_t vi = chunk_vec(c, clen, u);
        if (vi >= nvec) break;
        const uint64_t gi = vi * W;
        float g[W], p[W], m[W], v[W];
        if (SRC_WS) IO::ldf(a.ws.ghat, gi, g);
        else reduce_group<DT, IO>(a, gi, pro, g);
        IO::ldf(a.master + off, gi, p);
        IO::ldf(a.m + off, gi, m);
        IO::ldf(a.v + off, gi, v);
        const int valid = valid_count(gi, W, a.psi);
        uint32_t q[W];
#pragma unroll
        for (int k = 0; k < W; ++k) {
            if (k < valid) {
                const float gk = pro.use_clip ? __fmul_rn(g[k], pro.clip_f) : g[k];
                adam1(gk, p[k], m[k], v[k], pro.sc);
            } else {
                p[k] = 0.0f; m[k] = 0.0f; v[k] = 0.0f;
            }
            q[k] = narrow<DT>(p[k]);
        }
        IO::stf(a.master + off, gi, p);
        IO::stf(a.m + off, gi, m);
        IO::stf(a.v + off, gi, v);
        if (TO_SHARD) {
            IO::st16(a.params[0], gi, q);
        } else {
            for (int r = 0; r < a.n_ranks; ++r) IO::st16(a.params[r], gi, q);
        }
      }
      __syncthreads();
      ch.advance();
    }
}

// Stage 0, pass 2: every rank holds the full averaged gradient and its own
// full replica of master/m/v (rank r at r*psi_pad) and updates all of it.
template <int DT, class IO>
__global__ void __launch_bounds__(kThreads, 3) k_apply_stage0(const __grid_constant__ Args a) {
    pdl_enter();
    constexpr int W = IO::W;
    __shared__ Pro pro;
    __shared__ unsigned long long s_c[2];
    prologue_reduce(a, pro, false);
    if (pro.overflow) return;   // every CTA: the counter stays untouched
    const uint64_t nvec = a.count / W;
    const uint64_t clen = chunk_len(nvec), nchunks = chunk_total(nvec);
    const int U = chunk_u(nvec);
    ChunkCtr* ctr = a.ws.ctrs + a.ctr_slot;
    Chunks ch(ctr, s_c, nchunks);
    for (;;) {
      const uint64_t c = ch.current();
      if (c >= nchunks) break;
      ch.prefetch();
      for (int u = 0; u < U; ++u) {
        const uint64_t vi = chunk_vec(c, clen, u);
        if (vi >= nvec) break;
        const uint64_t gi = vi * W;
        float g[W];
        IO::ldf(a.ws.ghat, gi, g);
        const int valid = valid_count(gi, W, a.psi);
#pragma unroll
        for (int k = 0; k < W; ++k)
            if (k < valid && pro.use_clip) g[k] = __fmul_rn(g[k], pro.clip_f);
        for (int r = 0; r < a.n_ranks; ++r) {
            const uint64_t ri = static_cast<uint64_t>(r) * a.psi_pad + gi;
            float p[W], m[W], v[W];
            IO::ldf(a.master, ri, p);
            IO::ldf(a.m, ri, m);
            IO::ldf(a.v, ri, v);
            uint32_t q[W];
#pragma unroll
            for (int k = 0; k < W; ++k) {
                if (k < valid) {
                    adam1(g[k], p[k], m[k], v[k], pro.sc);
                } else {
                    p[k] = 0.0f; m[k] = 0.0f; v[k] = 0.0f;
                }
                q[k] = narrow<DT>(p[k]);
            }
            IO::stf(a.master, ri, p);
            IO::stf(a.m, ri, m);
            IO::stf(a.v, ri, v);
            IO::st16(a.params[r], gi, q);
        }
      }
      __syncthreads();
      ch.advance();
    }
}

// After a speculative pass: when the step overflowed, rewrite the 16-bit
// copies from the live (old) master; otherwise exit at once.
template <int DT, class IO, bool TO_SHARD>
__global__ void __launch_bounds__(kThreads) k_rollback(const __grid_constant__ Args a) {
    pdl_enter();
    constexpr int W = IO::W;
    __shared__ unsigned long long s_c[2];
    const DevStatus* st = a.ws.status;
    if (!st->overflow) return;   // every CTA: the counter stays untouched
    const uint64_t off = static_cast<uint64_t>(st->live_slot) * a.slot_stride;
    const uint64_t nvec = a.count / W;
    const uint64_t clen = chunk_len(nvec), nchunks = chunk_total(nvec);
    const int U = chunk_u(nvec);
    ChunkCtr* ctr = a.ws.ctrs + a.ctr_slot;
    Chunks ch(ctr, s_c, nchunks);
    for (;;) {
        const uint64_t c = ch.current();
        if (c >= nchunks) break;
        ch.prefetch();
        for (int u = 0; u < U; ++u) {
            const uint64_t vi = chunk_vec(c, clen, u);
            if (vi >= nvec) break;
            const uint64_t gi = a.base + vi * W;
            float p[W];
            IO::ldf(a.master + off, gi, p);
            uint32_t q[W];
#pragma unroll
            for (int k = 0; k < W; ++k) q[k] = narrow<DT>(p[k]);
            if (TO_SHARD) {
                IO::st16(a.params[0], gi, q);
            } else {
                for (int r = 0; r < a.n_ranks; ++r) IO::st16(a.params[r], gi, q);
            }
        }
        __syncthreads();
        ch.advance();
    }
}

// After k_step_spec (stages 1/2): on overflow, rewrite the replicas from the
// old master; when the step needs clipping, redo it from the old slot --
// reduce the N gradients again, scale by the clip factor, AdamW into the
// shadow slot, cast, all-gather -- for k_commit_redo to make live.
// Otherwise exit at once.
template <int DT, class IO>
__global__ void __launch_bounds__(kThreads) k_fixup(const __grid_constant__ Args a) {
    pdl_enter();
    constexpr int W = IO::W;
    __shared__ Pro pro;
    __shared__ unsigned long long s_c[2];
    prologue_reduce(a, pro, false);
    const DevStatus* st = a.ws.status;
    const int overflow = st->overflow, redo = st->redo;
    if (!overflow && !redo) return;   // every CTA: the counter stays untouched
    const uint64_t src = static_cast<uint64_t>(pro.live) * a.slot_stride;
    const uint64_t dst = static_cast<uint64_t>(pro.live ^ 1) * a.slot_stride;
    const uint64_t nvec = a.count / W;
    // a rollback restores only what the stopped pass may have written
    const uint64_t hw = st->hwm1;
    const uint64_t lim = (overflow && hw != 0 && hw - 1 < nvec) ? hw - 1 : nvec;
    const uint64_t clen = chunk_len(lim), nchunks = chunk_total(lim);
    const int U = chunk_u(lim);
    ChunkCtr* ctr = a.ws.ctrs + a.ctr_slot;
    Chunks ch(ctr, s_c, nchunks);
    for (;;) {
      const uint64_t c = ch.current();
      if (c >= nchunks) break;
      ch.prefetch();
      for (int u = 0; u < U; ++u) {
        const uint64_t vi = chunk_vec(c, clen, u);
        if (vi >= lim) break;
        const uint64_t gi = vi * W;
        float p[W];
        uint32_t q[W];
        IO::ldf(a.master + src, gi, p);
        if (overflow) {
#pragma unroll
            for (int k = 0; k < W; ++k) q[k] = narrow<DT>(p[k]);
        } else {
            float g[W], m[W], v[W];
            reduce_group<DT, IO>(a, gi, pro, g);
            IO::ldf(a.m + src, gi, m);
            IO::ldf(a.v + src, gi, v);
            const int valid = valid_count(gi, W, a.psi);
#pragma unroll
            for (int k = 0; k < W; ++k) {
                if (k < valid) {
                    adam1(__fmul_rn(g[k], pro.clip_f), p[k], m[k], v[k], pro.sc);
                } else {
                    p[k] = 0.0f; m[k] = 0.0f; v[k] = 0.0f;
                }
                q[k] = narrow<DT>(p[k]);
            }
            IO::stf(a.master + dst, gi, p);
            IO::stf(a.m + dst, gi, m);
            IO::stf(a.v + dst, gi, v);
        }
        for (int r = 0; r < a.n_ranks; ++r) IO::st16(a.params[r], gi, q);
      }
      __syncthreads();
      ch.advance();
    }
}

__global__ void k_commit_redo(DevStatus* st) {
    if (st->redo) {
        st->redo = 0;
        st->live_slot ^= 1;
        st->t += 1;
        st->applied = 1;
    }
    st->hwm1 = 0ull;
}

// ZeRO-3 gather of [base, base+count): out[r][j] = shard[base + j].
// 8-wide: a thread loads all its vectors of the chunk (up to kChunkU
// 16-byte loads in flight) before it stores them to the N outputs, and the
// grid is held at kGatherPerSm CTAs per SM.  Both measured faster than one
// load per store round on the full occupancy grid: this kernel writes N
// bytes for every byte it reads, and fewer, deeper streams suit that mix.
constexpr int kGatherPerSm = 3;

// One chunk c of an 8-wide gather of nvec vectors from src (starting at
// element base, a multiple of 8) to the n outputs.
__device__ __forceinline__ void gather_chunk8(const void* src, uint64_t base, void* const* outs, int n, uint64_t c,
                                              uint64_t clen, int U, uint64_t nvec) {
    static_assert(kChunkU == 4, "one batch of loads covers a chunk");
    uint4 x[kChunkU];
    uint64_t vi[kChunkU];
#pragma unroll
    for (int u = 0; u < kChunkU; ++u) {
        vi[u] = u < U ? chunk_vec(c, clen, u) : nvec;
        if (vi[u] < nvec) x[u] = __ldcs(reinterpret_cast<const uint4*>(src) + (base / 8 + vi[u]));
    }
    for (int r = 0; r < n; ++r) {
        uint4* out = reinterpret_cast<uint4*>(outs[r]);
#pragma unroll
        for (int u = 0; u < kChunkU; ++u)
            if (vi[u] < nvec) __stcs(out + vi[u], x[u]);
    }
}

template <class IO>
__global__ void __launch_bounds__(kThreads) k_gather(const __grid_constant__ Args a) {
    pdl_enter();
    constexpr int W = IO::W;
    __shared__ unsigned long long s_c[2];
    const uint64_t nvec = a.count / W;
    const uint64_t clen = chunk_len(nvec), nchunks = chunk_total(nvec);
    const int U = chunk_u(nvec);
    ChunkCtr* ctr = a.ws.ctrs + a.ctr_slot;
    Chunks ch(ctr, s_c, nchunks);
    for (;;) {
        const uint64_t c = ch.current();
        if (c >= nchunks) break;
        ch.prefetch();
        if constexpr (W == 8) {
            gather_chunk8(a.grads[0], a.base, a.params, a.n_ranks, c, clen, U, nvec);
        } else {
            for (int u = 0; u < U; ++u) {
                const uint64_t vi = chunk_vec(c, clen, u);
                if (vi >= nvec) break;
                const uint64_t j = vi * W;
                uint32_t x[W];
                IO::ld16(a.grads[0], a.base + j, x);
                for (int r = 0; r < a.n_ranks; ++r) IO::st16(a.params[r], j, x);
            }
        }
        __syncthreads();
        ch.advance();
    }
}

// Reduce-scatter of bucket [base, base+count) into the owners' shards
// (ZeRO-3; and ZeRO-2 when the gradients arrive bucket by bucket during
// backward).  SPEC: the bucket's AdamW update runs here into the shadow
// slot and its 16-bit result goes to the shard (stage 3) or to every
// rank's replica (TO_REPLICAS, stage 2); else g_hat goes to the workspace.
// The last block stores the bucket's norm partial and flag for the step's
// finaliser.
// Chunk cap of the reduce-scatter: with few ranks an iteration moves few
// bytes and longer chunks pay (16 measured 1.5-2 % faster at N = 2 and 4);
// from N = 8 up kChunkU measured better (shorter tail on 5e7-element buckets).
__host__ __device__ inline int rs_chunk_cap(int n_ranks) { return n_ranks <= 4 ? 16 : kChunkU; }
// Chunk target of the reduce-scatter: kRsReplicaChunks into the replicas;
// into the shard or the workspace, kRsSmallNChunks for N <= 2 and the
// default above.  At N = 2 a chunk of the default target lasts about 60 us
// on 5e7-element buckets, and the launch's last chunks leave SMs idle; at
// 4096 the stage-3 step at psi = 2^29 took 3.636 against 3.676 ms (6144:
// 3.647, 8192: 3.719), and at N = 4 it was slower (4.639 against 4.617 ms).
__host__ __device__ inline uint64_t rs_chunk_target(int n_ranks, bool to_replicas) {
    return to_replicas ? kRsReplicaChunks : (n_ranks <= kSmallN ? kRsSmallNChunks : kMinChunks);
}

// MINB as for the step: 4 CTAs per SM for N <= 2 (psi = 2^29, N = 2,
// 5e7-element buckets: 2.73 against 2.77 ms per step's reduce-scatters;
// slower from N = 4 up).
// GATHER (8-wide only): the launch's counter hands out the reduce-scatter's
// chunks, then the chunks of the gather of [gbase, gbase + gcount) of the
// 16-bit shard (params[0]) to gout[r], so that the CTAs that finish the
// reduce-scatter early go on to the gather instead of waiting for the
// launch's last chunks.  The two ranges are disjoint (checked on the host),
// so the result is that of the two calls one after the other.
template <int DT, class IO, bool SPEC, bool TO_REPLICAS, int MINB, bool GATHER>
__global__ void __launch_bounds__(kThreads, MINB) k_rs(const __grid_constant__ Args a) {
    pdl_enter();
    constexpr int W = IO::W;
    static_assert(!GATHER || W == 8, "the fused gather runs 8-wide");
    __shared__ Pro pro;
    __shared__ unsigned long long s_c[2];
    __shared__ double s_wp[2][kThreads / 32];
    prologue_reduce(a, pro, SPEC);
    const uint64_t src = static_cast<uint64_t>(pro.live) * a.slot_stride;
    const uint64_t dst = static_cast<uint64_t>(pro.live ^ 1) * a.slot_stride;
    const uint64_t nvec = a.count / W;
    const int umax = rs_chunk_cap(a.n_ranks);
    const uint64_t target = rs_chunk_target(a.n_ranks, TO_REPLICAS);
    const uint64_t clen = chunk_len(nvec, umax, target), nchunks = chunk_total(nvec, umax, target);
    const int U = chunk_u(nvec, umax, target);
    // the gather's chunks follow the reduce-scatter's (none unless GATHER);
    // its chunk geometry is formed again in its branch from the arguments,
    // so that it holds no registers across the reduce-scatter's loop
    const uint64_t ntotal = nchunks + (GATHER ? chunk_total(a.gcount / 8) : 0);
    ChunkCtr* ctr = a.ws.ctrs + a.ctr_slot;
    int bad = 0;
    Chunks ch(ctr, s_c, ntotal);
    for (;;) {
      const uint64_t c = ch.current();
      if (c >= nchunks) break;     // done, or the first of this CTA's gather chunks
      ch.prefetch();
      double acc = 0.0;
      for (int u = 0; u < U; ++u) {
        const uint64_t vi = chunk_vec(c, clen, u);
        if (vi >= nvec) break;
        const uint64_t j = vi * W;
        const uint64_t gi = a.base + j;
        float g[W];
        reduce_group<DT, IO>(a, j, pro, g);
        const int valid = valid_count(gi, W, a.psi);
        if (SPEC) {
            float p[W], m[W], v[W];
            IO::ldf(a.master + src, gi, p);
            IO::ldf(a.m + src, gi, m);
            IO::ldf(a.v + src, gi, v);
            norm_group<W>(g, valid, acc, bad);
            uint32_t q[W];
#pragma unroll
            for (int k = 0; k < W; ++k) {
                if (k < valid) {
                    adam1(g[k], p[k], m[k], v[k], pro.sc);
                } else {
                    p[k] = 0.0f; m[k] = 0.0f; v[k] = 0.0f;
                }
                q[k] = narrow<DT>(p[k]);
            }
            IO::stf(a.master + dst, gi, p);
            IO::stf(a.m + dst, gi, m);
            IO::stf(a.v + dst, gi, v);
            if (TO_REPLICAS) {
                for (int r = 0; r < a.n_ranks; ++r) IO::st16(a.params[r], gi, q);
            } else {
                IO::st16(a.params[0], gi, q);
            }
        } else {
            norm_group<W>(g, valid, acc, bad);
#pragma unroll
            for (int k = 0; k < W; ++k)
                if (k >= valid) g[k] = 0.0f;
            IO::stf(a.ws.ghat, gi, g);
        }
      }
      close_chunk(a.ws, c, nchunks, acc, s_wp, ch.parity(), 0);
      ch.advance();
    }
    if (GATHER) {
        // chunks are handed out in order: once a CTA holds a gather chunk it
        // gets no more reduce-scatter chunks
        const uint64_t gvec = a.gcount / 8, gclen = chunk_len(gvec);
        const int gU = chunk_u(gvec);
        for (;;) {
            const uint64_t c = ch.current();
            if (c >= ntotal) break;
            ch.prefetch();
            gather_chunk8(a.params[0], a.gbase, a.gout, a.n_ranks, c - nchunks, gclen, gU, gvec);
            __syncthreads();
            ch.advance();
        }
    }
    const int flag = __syncthreads_or(bad);
    if (publish(a, 0.0, flag, a.ws.partials, a.ws.flags)) {
        double qsum;
        int f;
        gather_groups(a.ws, nchunks, gridDim.x, qsum, f);
        if (threadIdx.x == 0) {
            ctr->next = 0ull;
            a.ws.bucket_norm[a.bucket_index] = qsum;
            a.ws.bucket_flag[a.bucket_index] = f;
            a.ws.status->ticket = 0u;
        }
    }
}

// ZeRO-3 step finaliser (one block): combine the buckets' partials in call
// order, then commit / skip (SPEC) or decide clip and scalars (two-pass).
template <bool SPEC>
__global__ void __launch_bounds__(kThreads) k_finalize3(const __grid_constant__ Args a) {
    pdl_enter();
    double q;
    int f;
    gather_partials(a.ws.bucket_norm, a.ws.bucket_flag, a.bucket_index, q, f);
    if (threadIdx.x == 0) {
        DevStatus* st = a.ws.status;
        if (f) status_skip(st, q);
        else if (SPEC) status_commit_spec(st, q);
        else status_decide_two_pass(st, q, a.hyper);
        // the next step's reduce-scatters (one per bucket) read these
        // instead of computing them in every CTA of every launch
        cache_next_scalars(st, a.hyper);
    }
}

__global__ void k_set_scaler(DevStatus* st, float loss_scale, int64_t t, int32_t slot) {
    st->loss_scale = loss_scale;
    st->t = t;
    st->live_slot = slot;
    st->skipped = 0;
    st->overflow = 0;
    st->applied = 0;
    st->norm = 0.0;
    st->clip_coef = 1.0;
    st->clip_f = 1.0f;
    st->use_clip = 0;
    st->error = 0;
    st->redo = 0;
    st->ticket = 0u;
    st->stop = 0u;
    st->hwm1 = 0ull;
    st->sc_t = -1;
}

// ------------------------------------------------------------------ launch
template <int DT, class IO>
cudaError_t launch_dw(Kind kind, const Args& a, cudaStream_t s, int* grid_out) {
    const uint64_t nvec = a.count / IO::W;
    switch (kind) {
        case Kind::kStepSpec:
            return a.n_ranks <= kSmallN
                       ? run_chunked_u(k_step_spec<DT, IO, 4>, a, nvec, kStepChunkU, step_chunk_target(a.n_ranks), s,
                                       grid_out)
                       : run_chunked_u(k_step_spec<DT, IO, 3>, a, nvec, kStepChunkU, step_chunk_target(a.n_ranks), s,
                                       grid_out);
        case Kind::kReduceWs: return run_chunked<kChunkU, kTwoPassChunks>(k_reduce<DT, IO, true>, a, nvec, s, grid_out);
        case Kind::kReduceNoWs: return run_chunked<kChunkU, kTwoPassChunks>(k_reduce<DT, IO, false>, a, nvec, s, grid_out);
        case Kind::kApplyWs: return run_chunked<kChunkU, kTwoPassChunks>(k_apply<DT, IO, true, false>, a, nvec, s, grid_out);
        case Kind::kApplyReread: return run_chunked<kChunkU, kTwoPassChunks>(k_apply<DT, IO, false, false>, a, nvec, s, grid_out);
        case Kind::kApplyWsShard: return run_chunked<kChunkU, kTwoPassChunks>(k_apply<DT, IO, true, true>, a, nvec, s, grid_out);
        case Kind::kApplyStage0: return run_chunked(k_apply_stage0<DT, IO>, a, nvec, s, grid_out);
        case Kind::kRollbackReplicas: return run_chunked(k_rollback<DT, IO, false>, a, nvec, s, grid_out);
        case Kind::kRollbackShard: return run_chunked(k_rollback<DT, IO, true>, a, nvec, s, grid_out);
        case Kind::kFixupReplicas: return run_chunked(k_fixup<DT, IO>, a, nvec, s, grid_out);
        case Kind::kGather: return run_chunked(k_gather<IO>, a, nvec, s, grid_out, IO::W == 8 ? kGatherPerSm : 0);
        case Kind::kRsSpec:
            return a.n_ranks <= kSmallN
                       ? run_chunked_u(k_rs<DT, IO, true, false, 4, false>, a, nvec, rs_chunk_cap(a.n_ranks),
                                       rs_chunk_target(a.n_ranks, false), s, grid_out)
                       : run_chunked_u(k_rs<DT, IO, true, false, 3, false>, a, nvec, rs_chunk_cap(a.n_ranks),
                                       rs_chunk_target(a.n_ranks, false), s, grid_out);
        case Kind::kRsSpecReplicas: return run_chunked_u(k_rs<DT, IO, true, true, 3, false>, a, nvec, rs_chunk_cap(a.n_ranks), rs_chunk_target(a.n_ranks, true), s,
                                                            grid_out);
        case Kind::kRsWs: return run_chunked_u(k_rs<DT, IO, false, false, 3, false>, a, nvec, rs_chunk_cap(a.n_ranks), rs_chunk_target(a.n_ranks, false), s, grid_out);
        case Kind::kRsSpecGather:
        case Kind::kRsWsGather:
            if constexpr (IO::W != 8) {
                return cudaErrorInvalidValue;
            } else {
                // one CTA per chunk at most, over both parts of the launch
                const uint64_t n = chunk_total(nvec, rs_chunk_cap(a.n_ranks), rs_chunk_target(a.n_ranks, false)) + chunk_total(a.gcount / 8);
                if (kind == Kind::kRsWsGather) return run(k_rs<DT, IO, false, false, 3, true>, a, n * kThreads, s, grid_out);
                return a.n_ranks <= kSmallN ? run(k_rs<DT, IO, true, false, 4, true>, a, n * kThreads, s, grid_out)
                                            : run(k_rs<DT, IO, true, false, 3, true>, a, n * kThreads, s, grid_out);
            }
    }
    return cudaErrorInvalidValue;
}

template <int DT>
cudaError_t launch_d(Kind kind, Vec vec, const Args& a, cudaStream_t s, int* grid_out) {
    switch (vec) {
        case Vec::k8s32: return launch_dw<DT, Io8s32>(kind, a, s, grid_out);
        case Vec::k8s16: return launch_dw<DT, Io8s16>(kind, a, s, grid_out);
        default: return launch_dw<DT, Io1>(kind, a, s, grid_out);
    }
}

}  // namespace

cudaError_t launch(Kind kind, int dtype, Vec vec, const Args& a, cudaStream_t s, int* grid_out) {
    return dtype == kFp16 ? launch_d<kFp16>(kind, vec, a, s, grid_out) : launch_d<kBf16>(kind, vec, a, s, grid_out);
}

cudaError_t launch_finalize3(bool spec, const Args& a, cudaStream_t s) {
    if (spec) k_finalize3<true><<<1, kThreads, 0, s>>>(a);
    else k_finalize3<false><<<1, kThreads, 0, s>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_commit_redo(DevStatus* st, cudaStream_t s) {
    k_commit_redo<<<1, 1, 0, s>>>(st);
    return cudaGetLastError();
}

cudaError_t launch_set_scaler(DevStatus* st, float loss_scale, int64_t t, int32_t slot, cudaStream_t s) {
    k_set_scaler<<<1, 1, 0, s>>>(st, loss_scale, t, slot);
    return cudaGetLastError();
}

}  // namespace zg
