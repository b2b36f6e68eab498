// The stage 1/2 speculative step with its inputs staged through shared
// memory by the bulk-copy engine (cp.async.bulk, completion on mbarriers).
//
// Same method and arithmetic as k_step_spec (zero_kernels.cu): N-rank
// reduce in rank order, unscale, overflow flag, norm partial, AdamW from
// the live slot into the shadow slot, RNE cast, all-gather to N replicas,
// last-block finalise.  What differs is how the inputs reach the SM: each
// CTA walks tiles of 2048 elements; per tile the N ranks' 16-bit gradient
// rows (4 KiB each) and the live slot's master/m/v rows (8 KiB each) are
// copied by one thread with bulk async copies into a ring of shared-memory
// stages, several tiles ahead of the computation, so the loads need no
// registers and no per-thread load instructions.  Outputs are written from
// registers with 256-bit (fp32) and 128-bit (16-bit) stores.
//
// Warp 8 issues the copies; warps 0-7 compute.
//
// Every mbarrier wait is bounded (2^24 polls and 2 s of %globaltimer).  A
// wait that gives up makes its CTA stop, wait -- again bounded -- for the
// copies it issued, set the device error word and flag the step as aborted:
// nothing is committed, the replicas are restored by k_fixup, and the loss
// scale is kept.

#include "zero_device.cuh"

namespace zg {
namespace {

constexpr int kTile = kThreads * 8;          // 2048 elements per tile
constexpr uint32_t kWaitIters = 1u << 24;
constexpr uint64_t kWaitNs = 2000000000ull;  // 2 s

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ bool mbar_test(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}
// Bounded wait for the phase of parity `parity` to complete.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity) {
    if (mbar_test(bar, parity)) return true;
    const uint64_t t0 = global_ns();
    for (uint32_t i = 0; i < kWaitIters; ++i) {
        if (mbar_test(bar, parity)) return true;
        if ((i & 255u) == 255u && global_ns() - t0 > kWaitNs) break;
    }
    return false;
}
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                 ::"r"(dst), "l"(src), "r"(bytes), "r"(bar)
                 : "memory");
}

// In the last block: the fixed-order sum of the blocks' partials (as
// gather_partials) and the OR of their flag bits.
__device__ void gather_flag_bits(const double* slot_norm, const int32_t* slot_flag, int count, double& q,
                                 int& bits) {
    __shared__ int s_bits;
    if (threadIdx.x == 0) s_bits = 0;
    __threadfence();
    __syncthreads();
    double s = 0.0;
    int f = 0;
    for (int b = threadIdx.x; b < count; b += blockDim.x) {
        s = __dadd_rn(s, *reinterpret_cast<const volatile double*>(slot_norm + b));
        f |= *reinterpret_cast<const volatile int32_t*>(slot_flag + b);
    }
    q = block_sum(s);
    if (f) atomicOr(&s_bits, f);
    __syncthreads();
    bits = s_bits;
}

// A wait gave up: the step is skipped like an overflowed one (state
// untouched, replicas restored by the fixup kernel, t not advanced) but the
// loss scale is kept; the device error word stays set.
__device__ void status_abort(DevStatus* st, double q) {
    st->overflow = 1;
    st->applied = 0;
    st->norm = __dsqrt_rn(q);
    st->clip_coef = 1.0;
    st->clip_f = 1.0f;
    st->use_clip = 0;
    st->skipped += 1;
}

struct TmaLayout {
    int stages;
    uint32_t stage_bytes;   // N*4096 + 3*8192
};

constexpr int kConsumerWarps = kThreads / 32;     // 8 warps compute
constexpr int kTmaThreads = kThreads + 32;        // + 1 producer warp

// Dynamic shared memory: [stages][N grad rows | master | m | v], then
// 2*stages mbarriers (full, empty).  Warps 0-7 compute; warp 8 (one lane)
// issues the copies, `stages` tiles ahead.
template <int DT>
__global__ void __launch_bounds__(kTmaThreads, 2) k_step_tma(const __grid_constant__ Args a, TmaLayout lay) {
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ Pro pro;
    __shared__ int abort_flag;
    __shared__ unsigned long long issued_total;
    prologue_reduce(a, pro, true);
    const int n = a.n_ranks;
    const uint32_t gbytes = kTile * 2, fbytes = kTile * 4;
    unsigned char* bars_base = smem + static_cast<size_t>(lay.stages) * lay.stage_bytes;
    const uint32_t full0 = smem_addr(bars_base), empty0 = full0 + 8 * lay.stages;
    if (threadIdx.x == 0) {
        abort_flag = 0;
        issued_total = 0ull;
        for (int s = 0; s < lay.stages; ++s) {
            mbar_init(full0 + 8 * s, 1);
            mbar_init(empty0 + 8 * s, kConsumerWarps);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();

    const uint64_t src_off = static_cast<uint64_t>(pro.live) * a.slot_stride;
    const uint64_t dst_off = static_cast<uint64_t>(pro.live ^ 1) * a.slot_stride;
    const uint64_t ntiles = a.count / kTile;
    // this CTA's tiles: blockIdx.x, blockIdx.x + gridDim.x, ...
    const uint64_t my_tiles = ntiles > blockIdx.x ? (ntiles - 1 - blockIdx.x) / gridDim.x + 1 : 0;
    volatile int* vabort = &abort_flag;

    double acc = 0.0;
    int bad = 0, aborted = 0;
    if (threadIdx.x >= kThreads) {
        // producer warp: lane 0 fills stage k % stages with tile k once the
        // consumers have released its previous fill
        if (threadIdx.x == kThreads) {
            uint64_t k = 0;
            for (; k < my_tiles; ++k) {
                if (*vabort) break;
                if (blockIdx.x == 0 && k + 1 == a.hold_tile1) break;   // held: the consumers' waits run out
                const int s = static_cast<int>(k % lay.stages);
                if (k >= static_cast<uint64_t>(lay.stages) &&
                    !mbar_wait(empty0 + 8 * s, static_cast<uint32_t>((k / lay.stages - 1) & 1))) {
                    *vabort = 1;
                    break;
                }
                const uint64_t e0 = (blockIdx.x + k * gridDim.x) * static_cast<uint64_t>(kTile);
                unsigned char* st = smem + static_cast<size_t>(s) * lay.stage_bytes;
                const uint32_t bar = full0 + 8 * s;
                mbar_expect_tx(bar, lay.stage_bytes);
                for (int r = 0; r < n; ++r)
                    bulk_g2s(smem_addr(st + r * gbytes), static_cast<const unsigned short*>(a.grads[r]) + e0, gbytes,
                             bar);
                unsigned char* sf = st + static_cast<size_t>(n) * gbytes;
                bulk_g2s(smem_addr(sf), a.master + src_off + e0, fbytes, bar);
                bulk_g2s(smem_addr(sf + fbytes), a.m + src_off + e0, fbytes, bar);
                bulk_g2s(smem_addr(sf + 2 * fbytes), a.v + src_off + e0, fbytes, bar);
            }
            issued_total = k;
        }
    } else {
        const int t = threadIdx.x;
        for (uint64_t k = 0; k < my_tiles; ++k) {
            const int s = static_cast<int>(k % lay.stages);
            const bool ok = mbar_wait(full0 + 8 * s, static_cast<uint32_t>((k / lay.stages) & 1));
            // leave together, warp by warp: no warp-collective op below may miss a lane
            if (__any_sync(0xFFFFFFFFu, !ok || *vabort)) {
                if ((t & 31) == 0) *vabort = 1;
                break;
            }
            const unsigned char* st = smem + static_cast<size_t>(s) * lay.stage_bytes;
            const uint64_t gi = (blockIdx.x + k * gridDim.x) * static_cast<uint64_t>(kTile) + 8 * t;
            // rank sum in order from +0
            float g[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) g[e] = 0.0f;
            for (int r = 0; r < n; ++r) {
                const uint4 x = *reinterpret_cast<const uint4*>(st + r * gbytes + 16 * t);
                const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    g[2 * e] = __fadd_rn(g[2 * e], widen<DT>(w[e] & 0xFFFFu));
                    g[2 * e + 1] = __fadd_rn(g[2 * e + 1], widen<DT>(w[e] >> 16));
                }
            }
#pragma unroll
            for (int e = 0; e < 8; ++e) g[e] = pro.use_div ? __fdiv_rn(g[e], pro.den) : __fmul_rn(g[e], pro.inv);
            float p[8], m[8], v[8];
            {
                const float4* s4 = reinterpret_cast<const float4*>(st + static_cast<size_t>(n) * gbytes);
                const float4 p0 = s4[2 * t], p1 = s4[2 * t + 1];
                const float4 m0 = s4[kTile / 4 + 2 * t], m1 = s4[kTile / 4 + 2 * t + 1];
                const float4 v0 = s4[kTile / 2 + 2 * t], v1 = s4[kTile / 2 + 2 * t + 1];
                p[0] = p0.x; p[1] = p0.y; p[2] = p0.z; p[3] = p0.w; p[4] = p1.x; p[5] = p1.y; p[6] = p1.z; p[7] = p1.w;
                m[0] = m0.x; m[1] = m0.y; m[2] = m0.z; m[3] = m0.w; m[4] = m1.x; m[5] = m1.y; m[6] = m1.z; m[7] = m1.w;
                v[0] = v0.x; v[1] = v0.y; v[2] = v0.z; v[3] = v0.w; v[4] = v1.x; v[5] = v1.y; v[6] = v1.z; v[7] = v1.w;
            }
            __syncwarp();
            if ((t & 31) == 0) mbar_arrive(empty0 + 8 * s);   // stage free for the next copies
            const int valid = valid_count(gi, 8, a.psi);
            norm_group<8>(g, valid, acc, bad);
            uint32_t q[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                if (e < valid) {
                    adam1(g[e], p[e], m[e], v[e], pro.sc);
                } else {
                    p[e] = 0.0f; m[e] = 0.0f; v[e] = 0.0f;
                }
                q[e] = narrow<DT>(p[e]);
            }
            Io8s32::stf(a.master + dst_off, gi, p);
            Io8s32::stf(a.m + dst_off, gi, m);
            Io8s32::stf(a.v + dst_off, gi, v);
            for (int r = 0; r < n; ++r) Io8s32::st16(a.params[r], gi, q);
        }
    }
    __syncthreads();
    if (abort_flag) {
        // leave no copy in flight: wait (bounded) for every stage this CTA filled
        if (threadIdx.x == kThreads) {
            const uint64_t issued = issued_total;
            for (int s = 0; s < lay.stages; ++s) {
                const uint64_t fills = issued > static_cast<uint64_t>(s) ? (issued - 1 - s) / lay.stages + 1 : 0;
                if (fills) mbar_wait(full0 + 8 * s, static_cast<uint32_t>((fills - 1) & 1));
            }
            atomicExch(&a.ws.status->error, 1);
        }
        aborted = 1;
    }
    // elements past the last full tile, element groups of 8 with plain loads
    {
        const Pro& pr = pro;
        for (uint64_t vi = ntiles * (kTile / 8) + thread_id(); vi < a.count / 8; vi += grid_threads()) {
            const uint64_t gi = vi * 8;
            float g[8], p[8], m[8], v[8];
            reduce_group<DT, Io8s32>(a, gi, pr, g);
            Io8s32::ldf(a.master + src_off, gi, p);
            Io8s32::ldf(a.m + src_off, gi, m);
            Io8s32::ldf(a.v + src_off, gi, v);
            const int valid = valid_count(gi, 8, a.psi);
            norm_group<8>(g, valid, acc, bad);
            uint32_t q[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                if (e < valid) {
                    adam1(g[e], p[e], m[e], v[e], pr.sc);
                } else {
                    p[e] = 0.0f; m[e] = 0.0f; v[e] = 0.0f;
                }
                q[e] = narrow<DT>(p[e]);
            }
            Io8s32::stf(a.master + dst_off, gi, p);
            Io8s32::stf(a.m + dst_off, gi, m);
            Io8s32::stf(a.v + dst_off, gi, v);
            for (int r = 0; r < n; ++r) Io8s32::st16(a.params[r], gi, q);
        }
    }
    const double blk = block_sum(acc);
    // bit 0: a non-finite gradient; bit 1: this CTA gave up a wait
    const int flag = (__syncthreads_or(bad) ? 1 : 0) | (__syncthreads_or(aborted) ? 2 : 0);
    if (publish(a, blk, flag, a.ws.partials, a.ws.flags)) {
        double qsum;
        int f;
        gather_flag_bits(a.ws.partials, a.ws.flags, gridDim.x, qsum, f);
        if (threadIdx.x == 0) {
            DevStatus* st = a.ws.status;
            if (f & 2) status_abort(st, qsum);
            else if (f) status_skip(st, qsum);
            else status_decide_spec(st, qsum, a.hyper);
            st->ticket = 0u;
        }
    }
}

}  // namespace

// Pipeline depth: as many stages of N*4 KiB + 24 KiB as fit in 112 KiB
// (two CTAs per SM), else in 200 KiB (one CTA per SM), at most 4; 0 when
// not even two fit.
namespace {
constexpr uint32_t kBudget2 = 112u * 1024u, kBudget1 = 200u * 1024u;
uint32_t tma_stage_bytes(int n_ranks) { return static_cast<uint32_t>(n_ranks) * kTile * 2 + 3u * kTile * 4; }
}  // namespace

int tma_stages(int n_ranks) {
    const uint32_t stage = tma_stage_bytes(n_ranks);
    int s = static_cast<int>(kBudget2 / stage);
    if (s < 2) s = static_cast<int>(kBudget1 / stage);
    return s >= 2 ? (s > 4 ? 4 : s) : 0;
}

cudaError_t launch_step_tma(int dtype, const Args& a, cudaStream_t s) {
    TmaLayout lay;
    lay.stages = tma_stages(a.n_ranks);
    lay.stage_bytes = tma_stage_bytes(a.n_ranks);
    if (lay.stages < 2) return cudaErrorInvalidValue;
    const size_t smem = static_cast<size_t>(lay.stages) * lay.stage_bytes + 16 * lay.stages;
    auto kern = dtype == kFp16 ? k_step_tma<kFp16> : k_step_tma<kBf16>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    int dev = 0, sms = 0, per_sm = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kTmaThreads, smem)) != cudaSuccess)
        return e;
    if (per_sm < 1) return cudaErrorInvalidConfiguration;
    const uint64_t ntiles = a.count / kTile;
    uint64_t grid = static_cast<uint64_t>(sms) * static_cast<uint64_t>(per_sm);
    if (grid > static_cast<uint64_t>(kMaxBlocks)) grid = kMaxBlocks;
    if (ntiles < grid) grid = ntiles > 0 ? ntiles : 1;
    kern<<<static_cast<unsigned>(grid), kTmaThreads, smem, s>>>(a, lay);
    return cudaGetLastError();
}

}  // namespace zg
