// Device helpers shared by the kernel translation units (zero_kernels.cu,
// zero_quant.cu): 16-bit conversions, vector I/O policies, the Adam update,
// the unscale prologue, norm partials, and the last-block reduction that
// replaces a scalar all-reduce.  Each translation unit gets its own copy
// (anonymous namespace).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <mutex>

#include "zero_internal.h"

namespace zg {
namespace {

// ------------------------------------------------------------------ 16-bit
template <int DT>
__device__ __forceinline__ float widen(uint32_t bits16);
template <>
__device__ __forceinline__ float widen<kFp16>(uint32_t b) {
    return __half2float(__ushort_as_half(static_cast<unsigned short>(b)));
}
template <>
__device__ __forceinline__ float widen<kBf16>(uint32_t b) {
    return __uint_as_float(b << 16);
}

template <int DT>
__device__ __forceinline__ uint32_t narrow(float x);
template <>
__device__ __forceinline__ uint32_t narrow<kFp16>(float x) {
    return __half_as_ushort(__float2half_rn(x));
}
template <>
__device__ __forceinline__ uint32_t narrow<kBf16>(float x) {
    return __bfloat16_as_ushort(__float2bfloat16_rn(x));
}

// Vector I/O policies.  An IO type moves IO::W consecutive elements per
// thread: 16-bit values (gradients, replicas) and fp32 values (master, m,
// v, g_hat).
//   Io8s32: 8 elements; 16-bit as one 128-bit access, fp32 as one 256-bit
//           access (ld/st.global.v8.f32, sm_100 and later; 32-byte aligned);
//   Io8s16: 8 elements; fp32 as two 128-bit accesses (16-byte aligned);
//   Io1:    one element (any size, any offset).
// All accesses carry the streaming hint (.cs): nothing is re-read within a step.
struct Io8s16 {
    static constexpr int W = 8;
    __device__ static __forceinline__ void ld16(const void* p, uint64_t i, uint32_t (&out)[8]) {
        const uint4 x = __ldcs(reinterpret_cast<const uint4*>(p) + (i >> 3));
        out[0] = x.x & 0xFFFFu; out[1] = x.x >> 16;
        out[2] = x.y & 0xFFFFu; out[3] = x.y >> 16;
        out[4] = x.z & 0xFFFFu; out[5] = x.z >> 16;
        out[6] = x.w & 0xFFFFu; out[7] = x.w >> 16;
    }
    __device__ static __forceinline__ void st16(void* p, uint64_t i, const uint32_t (&q)[8]) {
        uint4 x;
        x.x = q[0] | (q[1] << 16); x.y = q[2] | (q[3] << 16);
        x.z = q[4] | (q[5] << 16); x.w = q[6] | (q[7] << 16);
        __stcs(reinterpret_cast<uint4*>(p) + (i >> 3), x);
    }
    __device__ static __forceinline__ void ldf(const float* p, uint64_t i, float (&out)[8]) {
        const float4 a = __ldcs(reinterpret_cast<const float4*>(p + i));
        const float4 b = __ldcs(reinterpret_cast<const float4*>(p + i) + 1);
        out[0] = a.x; out[1] = a.y; out[2] = a.z; out[3] = a.w;
        out[4] = b.x; out[5] = b.y; out[6] = b.z; out[7] = b.w;
    }
    __device__ static __forceinline__ void stf(float* p, uint64_t i, const float (&x)[8]) {
        __stcs(reinterpret_cast<float4*>(p + i), make_float4(x[0], x[1], x[2], x[3]));
        __stcs(reinterpret_cast<float4*>(p + i) + 1, make_float4(x[4], x[5], x[6], x[7]));
    }
};

struct Io8s32 : Io8s16 {
    // one 256-bit access per thread: a warp covers 1 KiB contiguous in one instruction
    __device__ static __forceinline__ void ldf(const float* p, uint64_t i, float (&o)[8]) {
        asm("ld.global.cs.v8.f32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
            : "=f"(o[0]), "=f"(o[1]), "=f"(o[2]), "=f"(o[3]), "=f"(o[4]), "=f"(o[5]), "=f"(o[6]), "=f"(o[7])
            : "l"(p + i));
    }
    __device__ static __forceinline__ void stf(float* p, uint64_t i, const float (&x)[8]) {
        asm volatile("st.global.cs.v8.f32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};"
                     :: "l"(p + i), "f"(x[0]), "f"(x[1]), "f"(x[2]), "f"(x[3]), "f"(x[4]), "f"(x[5]),
                        "f"(x[6]), "f"(x[7])
                     : "memory");
    }
};

struct Io1 {
    static constexpr int W = 1;
    __device__ static __forceinline__ void ld16(const void* p, uint64_t i, uint32_t (&out)[1]) {
        out[0] = __ldcs(reinterpret_cast<const unsigned short*>(p) + i);
    }
    __device__ static __forceinline__ void st16(void* p, uint64_t i, const uint32_t (&q)[1]) {
        __stcs(reinterpret_cast<unsigned short*>(p) + i, static_cast<unsigned short>(q[0]));
    }
    __device__ static __forceinline__ void ldf(const float* p, uint64_t i, float (&out)[1]) {
        out[0] = __ldcs(p + i);
    }
    __device__ static __forceinline__ void stf(float* p, uint64_t i, const float (&x)[1]) {
        __stcs(p + i, x[0]);
    }
};

// ------------------------------------------------------------------ scalars
// Adam coefficients of step t, formed in double and rounded once to fp32.
// Two halves with one double pow() each, so that two threads can form them
// at once (an FP64 pow is a long dependent chain on GB300).
__device__ void scalars_b1_part(const HyperDev& h, int64_t t, StepScalars& s) {
    const double lr = h.lr, b1 = h.beta1, b2 = h.beta2, wd = h.weight_decay;
    const double bc1 = __dsub_rn(1.0, pow(b1, static_cast<double>(t)));
    s.b1 = h.beta1;
    s.b2 = h.beta2;
    s.a1 = __double2float_rn(__dsub_rn(1.0, b1));
    s.a2 = __double2float_rn(__dsub_rn(1.0, b2));
    s.eps = h.eps;
    s.dfac = __double2float_rn(__dsub_rn(1.0, __dmul_rn(lr, wd)));
    s.step_size = __double2float_rn(__ddiv_rn(lr, bc1));
}
__device__ float scalars_bc2s(const HyperDev& h, int64_t t) {
    const double b2 = h.beta2;
    const double bc2 = __dsub_rn(1.0, pow(b2, static_cast<double>(t)));
    return __double2float_rn(__dsqrt_rn(bc2));
}
__device__ StepScalars make_scalars(const HyperDev& h, int64_t t) {
    StepScalars s;
    scalars_b1_part(h, t, s);
    s.bc2s = scalars_bc2s(h, t);
    return s;
}

// One AdamW update, each operation rounded once, in the oracle's order.
__device__ __forceinline__ void adam1(float g, float& p, float& m, float& v, const StepScalars& c) {
    p = __fmul_rn(p, c.dfac);
    m = __fadd_rn(__fmul_rn(c.b1, m), __fmul_rn(c.a1, g));
    v = __fadd_rn(__fmul_rn(c.b2, v), __fmul_rn(c.a2, __fmul_rn(g, g)));
    const float den = __fadd_rn(__fdiv_rn(__fsqrt_rn(v), c.bc2s), c.eps);
    p = __fsub_rn(p, __fmul_rn(c.step_size, __fdiv_rn(m, den)));
}

__device__ __forceinline__ bool nonfinite(float x) {
    return (__float_as_uint(x) & 0x7F800000u) == 0x7F800000u;
}

// Per-block view of the device status, read once by thread 0.
struct Pro {
    StepScalars sc;
    float den, inv, clip_f;
    int use_div, live, use_clip, overflow;
};

// Prologue of kernels that reduce gradients: unscale denominator N*scale
// (fp32 product, as the oracle forms it) and, for the one-pass kernels,
// the Adam coefficients of step t+1.
// The status word holds the step scalars for (t + 1, these hyper-parameters).
__device__ __forceinline__ bool scalars_cached(const DevStatus* st, const HyperDev& h) {
    const HyperDev& k = st->sc_key;
    return st->sc_t == st->t + 1 && __float_as_uint(k.lr) == __float_as_uint(h.lr) &&
           __float_as_uint(k.beta1) == __float_as_uint(h.beta1) &&
           __float_as_uint(k.beta2) == __float_as_uint(h.beta2) &&
           __float_as_uint(k.eps) == __float_as_uint(h.eps) &&
           __float_as_uint(k.weight_decay) == __float_as_uint(h.weight_decay);
}

__device__ __forceinline__ void prologue_reduce(const Args& a, Pro& pro, bool with_scalars) {
    // not cached: thread 32 forms bc2s while thread 0 forms the rest
    if (with_scalars && threadIdx.x == 32) {
        const DevStatus* st = a.ws.status;
        if (!scalars_cached(st, a.hyper)) pro.sc.bc2s = scalars_bc2s(a.hyper, st->t + 1);
    }
    if (threadIdx.x == 0) {
        const DevStatus* st = a.ws.status;
        const float den = __fmul_rn(static_cast<float>(a.n_ranks), st->loss_scale);
        const uint32_t bits = __float_as_uint(den);
        const uint32_t ex = (bits >> 23) & 0xFFu;
        // a power of two whose reciprocal is a normal number: s*inv == s/den exactly
        const bool pow2 = (bits & 0x7FFFFFu) == 0u && ex >= 1u && ex <= 253u;
        pro.den = den;
        pro.use_div = pow2 ? 0 : 1;
        pro.inv = pow2 ? __fdiv_rn(1.0f, den) : 0.0f;
        pro.live = st->live_slot;
        pro.clip_f = st->clip_f;
        pro.use_clip = st->use_clip;
        pro.overflow = st->overflow;
        if (with_scalars) {
            if (scalars_cached(st, a.hyper)) pro.sc = st->sc_next;
            else scalars_b1_part(a.hyper, st->t + 1, pro.sc);
        } else {
            pro.sc = st->sc;
        }
    }
    __syncthreads();
}

// Sum of the N ranks' values of W elements at local index j, then unscale.
template <int DT, class IO>
__device__ __forceinline__ void reduce_group(const Args& a, uint64_t j, const Pro& pro, float (&g)[IO::W]) {
    constexpr int W = IO::W;
    float s[W];
#pragma unroll
    for (int k = 0; k < W; ++k) s[k] = 0.0f;
    const int n = a.n_ranks;
    int r = 0;
    for (; r + 8 <= n; r += 8) {
        uint32_t raw[8][W];
#pragma unroll
        for (int q = 0; q < 8; ++q) IO::ld16(a.grads[r + q], j, raw[q]);
#pragma unroll
        for (int q = 0; q < 8; ++q)
#pragma unroll
            for (int k = 0; k < W; ++k) s[k] = __fadd_rn(s[k], widen<DT>(raw[q][k]));
    }
    for (; r < n; ++r) {
        uint32_t raw[W];
        IO::ld16(a.grads[r], j, raw);
#pragma unroll
        for (int k = 0; k < W; ++k) s[k] = __fadd_rn(s[k], widen<DT>(raw[k]));
    }
#pragma unroll
    for (int k = 0; k < W; ++k) g[k] = pro.use_div ? __fdiv_rn(s[k], pro.den) : __fmul_rn(s[k], pro.inv);
}

// Squares of the real elements into the thread's fp64 accumulator: an
// exact product (FMA error term) and a compensated fp32 sum per group, then
// one fp64 add, so the result carries ~1e-14 relative error.  That holds
// while every square and the group's sum lie in fp32's normal range.  A
// group with an element of magnitude 2^60 or more (its sum may overflow),
// or whose largest nonzero magnitude is below 2^-60 (its squares would be
// subnormal or zero), is summed in fp64 instead, where the square of every
// fp32 value is exact.  Non-finite elements only raise `bad`.
template <int W>
__device__ __forceinline__ void norm_group(const float (&g)[W], int valid, double& acc, int& bad) {
    float hi = 0.0f, lo = 0.0f, amax = 0.0f;
#pragma unroll
    for (int k = 0; k < W; ++k) {
        if (k < valid) {
            const float x = g[k];
            bad |= nonfinite(x) ? 1 : 0;
            amax = fmaxf(amax, fabsf(x));
            const float p = __fmul_rn(x, x);
            const float e = __fmaf_rn(x, x, -p);
            const float s = __fadd_rn(hi, p);
            const float bp = __fsub_rn(s, hi);
            const float err = __fadd_rn(__fsub_rn(hi, __fsub_rn(s, bp)), __fsub_rn(p, bp));
            hi = s;
            lo = __fadd_rn(lo, __fadd_rn(err, e));
        }
    }
    if (!(amax < 0x1p60f) || (amax > 0.0f && amax < 0x1p-60f)) {
        double q = 0.0;
#pragma unroll
        for (int k = 0; k < W; ++k)
            if (k < valid) {
                const double x = static_cast<double>(g[k]);
                q = __dadd_rn(q, __dmul_rn(x, x));
            }
        acc = __dadd_rn(acc, q);
    } else {
        acc = __dadd_rn(acc, __dadd_rn(static_cast<double>(hi), static_cast<double>(lo)));
    }
}

__device__ __forceinline__ int valid_count(uint64_t gi, int W, uint64_t psi) {
    if (gi + W <= psi) return W;
    if (gi >= psi) return 0;
    return static_cast<int>(psi - gi);
}

// Deterministic block sum (fixed shuffle tree, then warp sums in order);
// any block size up to 1024 threads.
__device__ double block_sum(double x) {
    __shared__ double sm[32];
    __syncthreads();
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) x = __dadd_rn(x, __shfl_down_sync(0xFFFFFFFFu, x, off));
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (lane == 0) sm[warp] = x;
    __syncthreads();
    double t = 0.0;
    if (threadIdx.x == 0) {
        for (int w = 0; w < (int)(blockDim.x >> 5); ++w) t = __dadd_rn(t, sm[w]);
    }
    return t;  // valid in thread 0
}

// Publish the block's partial; true in every thread of the last block.
__device__ bool publish(const Args& a, double blk, int flag, double* slot_norm, int32_t* slot_flag) {
    __shared__ int s_last;
    if (threadIdx.x == 0) {
        slot_norm[blockIdx.x] = blk;
        slot_flag[blockIdx.x] = flag;
        __threadfence();
        const unsigned prev = atomicAdd(&a.ws.status->ticket, 1u);
        s_last = (prev == gridDim.x - 1) ? 1 : 0;
    }
    __syncthreads();
    return s_last != 0;
}

// In the last block: fixed-order sum of all blocks' partials.
__device__ void gather_partials(const double* slot_norm, const int32_t* slot_flag, int count,
                                double& q, int& flag) {
    __threadfence();
    double s = 0.0;
    int f = 0;
    for (int b = threadIdx.x; b < count; b += blockDim.x) {
        s = __dadd_rn(s, *reinterpret_cast<const volatile double*>(slot_norm + b));
        f |= *reinterpret_cast<const volatile int32_t*>(slot_flag + b);
    }
    q = block_sum(s);
    flag = __syncthreads_or(f);
}

// After a step is finalised: the next step's one-pass scalars, once, for
// the kernels' prologues (same function and inputs as there, so the same
// bits).
__device__ void cache_next_scalars(DevStatus* st, const HyperDev& h) {
    st->sc_next = make_scalars(h, st->t + 1);
    st->sc_key = h;
    st->sc_t = st->t + 1;
}

// Overflow: skip.  The scale halves (floor 1.0); t and the state stay.
__device__ void status_skip(DevStatus* st, double q) {
    st->overflow = 1;
    st->applied = 0;
    st->norm = __dsqrt_rn(q);
    st->clip_coef = 1.0;
    st->clip_f = 1.0f;
    st->use_clip = 0;
    st->loss_scale = fmaxf(__fmul_rn(st->loss_scale, 0.5f), 1.0f);
    st->skipped += 1;
}

// Speculative pass done without overflow: the shadow slot becomes live.
__device__ void status_commit_spec(DevStatus* st, double q) {
    st->overflow = 0;
    st->applied = 1;
    st->norm = __dsqrt_rn(q);
    st->clip_coef = 1.0;
    st->clip_f = 1.0f;
    st->use_clip = 0;
    st->live_slot ^= 1;
    st->t += 1;
}

// Speculative one-pass step done without overflow.  With no clipping
// needed the shadow slot becomes live; when the norm calls for clipping
// (max_norm > 0 and max_norm / (norm + 1e-6) < 1) the step is marked for a
// redo from the old slot with the clip factor and step t+1 scalars.
__device__ void status_decide_spec(DevStatus* st, double q, const HyperDev& h) {
    const double norm = __dsqrt_rn(q);
    if (h.max_norm > 0.0f) {
        const double c = __ddiv_rn(static_cast<double>(h.max_norm), __dadd_rn(norm, 1e-6));
        if (c < 1.0) {
            st->overflow = 0;
            st->applied = 0;
            st->norm = norm;
            st->use_clip = 1;
            st->clip_f = __double2float_rn(c);
            st->clip_coef = static_cast<double>(st->clip_f);
            st->redo = 1;
            st->sc = make_scalars(h, st->t + 1);
            return;
        }
    }
    status_commit_spec(st, q);
}

// Two-pass decision before the apply pass: clip factor and step t+1 scalars.
__device__ void status_decide_two_pass(DevStatus* st, double q, const HyperDev& h) {
    const double norm = __dsqrt_rn(q);
    st->overflow = 0;
    st->applied = 1;
    st->norm = norm;
    st->use_clip = 0;
    st->clip_f = 1.0f;
    if (h.max_norm > 0.0f) {
        const double c = __ddiv_rn(static_cast<double>(h.max_norm), __dadd_rn(norm, 1e-6));
        if (c < 1.0) {
            st->use_clip = 1;
            st->clip_f = __double2float_rn(c);
        }
    }
    st->clip_coef = static_cast<double>(st->clip_f);
    st->t += 1;
    st->sc = make_scalars(h, st->t);
}

__device__ __forceinline__ uint64_t grid_threads() {
    return static_cast<uint64_t>(gridDim.x) * blockDim.x;
}
__device__ __forceinline__ uint64_t thread_id() {
    return static_cast<uint64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
}

// ------------------------------------------------------------ dynamic chunks
// The CTAs of a persistent grid do not progress at one rate: with a static
// grid-stride assignment the fast ones finish early and the launch ends in a
// tail where only the slow ones stream (about 7 % of the step on a GB300).
// Chunked kernels instead take chunk after chunk from their launch's counter;
// thread 0 fetches the next index while the block works on the current one.
// With U = chunk_u(nvec), thread t of whichever CTA takes chunk c handles the
// vectors c*U*kThreads + u*kThreads + t, u < U.
class Chunks {
  public:
    // A CTA's first chunk is its own index (the grid has no more CTAs than
    // chunks); each chunk it works on, thread 0 grabs the next from the
    // counter, which hands out gridDim.x, gridDim.x + 1, ...  So a launch
    // makes exactly nchunks grabs, and the CTA that makes grab nchunks - 1
    // (its failing one, like every CTA's last) resets the counter: every
    // other grab of the launch came before it.
    __device__ Chunks(ChunkCtr* ctr, unsigned long long* s2, uint64_t nchunks)
        : ctr_(ctr), s_(s2), n_(nchunks), par_(0), first_(true) {}
    __device__ uint64_t current() const { return first_ ? static_cast<uint64_t>(blockIdx.x) : s_[par_]; }
    __device__ int parity() const { return par_; }
    // thread 0, at the start of each chunk's work (nothing to grab when
    // every CTA has at most its own chunk)
    __device__ void prefetch() {
        if (threadIdx.x == 0) {
            if (n_ <= gridDim.x) {
                s_[par_ ^ 1] = ~0ull;
                return;
            }
            const unsigned long long v = atomicAdd(&ctr_->next, 1ull);
            if (v + 1 == n_) atomicExch(&ctr_->next, 0ull);
            s_[par_ ^ 1] = static_cast<unsigned long long>(gridDim.x) + v;
        }
    }
    // after the block barrier that closes a chunk
    __device__ void advance() {
        par_ ^= 1;
        first_ = false;
    }

  private:
    ChunkCtr* ctr_;
    unsigned long long* s_;
    uint64_t n_;
    int par_;
    bool first_;
};

// vector u of this thread in chunk c (chunks of `len` = U * kThreads vectors)
__device__ __forceinline__ uint64_t chunk_vec(uint64_t c, uint64_t len, int u) {
    return c * len + static_cast<uint64_t>(u) * kThreads + threadIdx.x;
}

__device__ __forceinline__ uint64_t group_count(uint64_t nchunks) { return (nchunks + kGroup - 1) / kGroup; }

// Fixed-order warp sum of doubles (lane 0 holds the result).
__device__ __forceinline__ double warp_dsum(double x) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) x = __dadd_rn(x, __shfl_down_sync(0xFFFFFFFFu, x, off));
    return x;
}

// Warp 0, after the barrier that closes chunk c: the chunk's norm partial is
// the sum, in warp order, of the warps' sums wp[] (each a fixed warp tree over
// the lanes' accumulators, written before the barrier).  The CTA that
// completes a group of kGroup chunks sums the group with a fixed tree.  None
// of this depends on which CTA took which chunk.
__device__ void commit_chunk(const Workspace& ws, uint64_t c, uint64_t nchunks, const double* wp) {
    const int lane = threadIdx.x & 31;
    const uint64_t g = c / kGroup;
    const uint64_t c0 = g * kGroup;
    const uint32_t members = static_cast<uint32_t>(nchunks - c0 < kGroup ? nchunks - c0 : kGroup);
    const bool grouped = nchunks > kDirectChunks;   // else the finaliser sums the chunks
    int last = 0;
    if (lane == 0) {
        double s = 0.0;
        for (int w = 0; w < kThreads / 32; ++w) s = __dadd_rn(s, wp[w]);
        ws.chunk_part[c] = s;
        if (grouped) {
            __threadfence();
            last = atomicAdd(&ws.group_ticket[g], 1u) == members - 1 ? 1 : 0;
        }
    }
    last = __shfl_sync(0xFFFFFFFFu, last, 0);
    if (last) {
        __threadfence();
        double x = static_cast<uint32_t>(lane) < members
                       ? *reinterpret_cast<const volatile double*>(ws.chunk_part + c0 + lane)
                       : 0.0;
        x = warp_dsum(x);
        if (lane == 0) {
            ws.group_part[g] = x;
            ws.group_ticket[g] = 0u;
        }
    }
}

// The chunk's closing barrier with its norm partial: each warp's sum goes to
// s_wp[parity], the barrier ORs `leave_in`, then warp 0 commits the chunk.
__device__ __forceinline__ int close_chunk(const Workspace& ws, uint64_t c, uint64_t nchunks, double cacc,
                                           double (*s_wp)[kThreads / 32], int parity, int leave_in) {
    const double w = warp_dsum(cacc);
    if ((threadIdx.x & 31) == 0) s_wp[parity][threadIdx.x >> 5] = w;
    const int leave = __syncthreads_or(leave_in);
    if (threadIdx.x < 32) commit_chunk(ws, c, nchunks, s_wp[parity]);
    return leave;
}

// In the finalising CTA of a chunked launch: fixed-order sum of the group
// partials (or, up to kDirectChunks chunks, of the chunk partials), and the
// OR of the CTAs' flags.
__device__ void gather_groups(const Workspace& ws, uint64_t nchunks, int nblocks, double& q, int& flag) {
    __threadfence();
    const bool grouped = nchunks > kDirectChunks;
    const double* part = grouped ? ws.group_part : ws.chunk_part;
    const uint64_t n = grouped ? group_count(nchunks) : nchunks;
    double s = 0.0;
    int f = 0;
    for (uint64_t g = threadIdx.x; g < n; g += blockDim.x)
        s = __dadd_rn(s, *reinterpret_cast<const volatile double*>(part + g));
    for (int b = threadIdx.x; b < nblocks; b += blockDim.x) f |= *reinterpret_cast<const volatile int32_t*>(ws.flags + b);
    q = block_sum(s);
    flag = __syncthreads_or(f);
}

// A pass cut short leaves groups with missing chunks: the finalising CTA
// zeroes their tickets.
__device__ void reset_groups(const Workspace& ws, uint64_t nchunks) {
    if (nchunks <= kDirectChunks) return;
    const uint64_t ngroups = group_count(nchunks);
    for (uint64_t g = threadIdx.x; g < ngroups; g += blockDim.x) ws.group_ticket[g] = 0u;
}

// Programmatic dependent launch.  run() launches every kernel with
// programmatic stream serialisation, so the next kernel in the stream may be
// scheduled before this one has finished.  Every kernel launched through
// run() therefore begins with pdl_enter(): it waits until the previous grid
// in the stream has completed and its memory is visible (a no-op when the
// kernel was not launched that way), and only then lets the next grid be
// scheduled.  The next grid's CTAs take SM slots as this grid's CTAs leave
// and wait there, which hides the launch latency between the kernels of a
// step; no two kernels' memory accesses ever overlap.
__device__ __forceinline__ void pdl_enter() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// CTAs of `kernel` resident at once on device `dev` (SMs x CTAs per SM, the
// latter capped at per_sm when per_sm > 0), with the occupancy queried once
// per kernel and device: the query costs more host time than a small launch.
template <typename KernelT>
cudaError_t resident_ctas(KernelT kernel, int dev, int per_sm_cap, uint64_t* out) {
    struct Entry {
        const void* kernel;
        int dev;
        int sms;
        int per_sm;
    };
    static Entry cache[512];
    static int used = 0;
    static std::mutex mu;
    std::lock_guard<std::mutex> lock(mu);
    int sms = 0, per_sm = 0;
    bool found = false;
    for (int i = 0; i < used; ++i)
        if (cache[i].kernel == reinterpret_cast<const void*>(kernel) && cache[i].dev == dev) {
            sms = cache[i].sms;
            per_sm = cache[i].per_sm;
            found = true;
            break;
        }
    if (!found) {
        cudaError_t e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, kThreads, 0);
        if (e != cudaSuccess) return e;
        if (per_sm < 1) per_sm = 1;
        if (used < 512) cache[used++] = Entry{reinterpret_cast<const void*>(kernel), dev, sms, per_sm};
    }
    if (per_sm_cap > 0 && per_sm > per_sm_cap) per_sm = per_sm_cap;
    *out = static_cast<uint64_t>(sms) * static_cast<uint64_t>(per_sm);
    return cudaSuccess;
}

// Launch on a persistent grid: as many CTAs as fit on the SMs at once (from
// the occupancy API, or per_sm CTAs per SM when per_sm > 0 caps it lower),
// or fewer when `nvec` vectors need fewer, capped at the per-block partial
// slots.  The kernel must begin with pdl_enter() (see above).
template <typename KernelT>
cudaError_t run(KernelT kernel, const Args& a, uint64_t nvec, cudaStream_t s, int* grid_out, int per_sm = 0) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    uint64_t cap = 0;
    if ((e = resident_ctas(kernel, dev, per_sm, &cap)) != cudaSuccess) return e;
    uint64_t want = (nvec + kThreads - 1) / kThreads;
    if (cap > static_cast<uint64_t>(kMaxBlocks)) cap = kMaxBlocks;
    uint64_t grid = want < cap ? want : cap;
    if (grid < 1) grid = 1;
    if (grid_out) *grid_out = static_cast<int>(grid);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, a);
}

// Launch a chunked kernel: the persistent grid, but no more CTAs than chunks.
template <int UMAX = kChunkU, uint64_t TARGET = kMinChunks, typename KernelT>
cudaError_t run_chunked(KernelT kernel, const Args& a, uint64_t nvec, cudaStream_t s, int* grid_out,
                        int per_sm = 0) {
    return run(kernel, a, chunk_total<UMAX, TARGET>(nvec) * kThreads, s, grid_out, per_sm);
}
// The same with the chunk cap and target chosen at run time (the kernel
// computes the same pair from its arguments).
template <typename KernelT>
cudaError_t run_chunked_u(KernelT kernel, const Args& a, uint64_t nvec, int umax, uint64_t target,
                          cudaStream_t s, int* grid_out) {
    return run(kernel, a, chunk_total(nvec, umax, target) * kThreads, s, grid_out);
}

}  // namespace
}  // namespace zg
