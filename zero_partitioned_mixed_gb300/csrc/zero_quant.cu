// ZeRO++ block-quantized exchanges for sm_103a.
//
// "CMU 11-868 L18" notes, other memory optimizations (ZeRO++): parameters
// are block-quantized from 16 bits to INT8 with zero-point quantization for
// the forward gather (qwZ), and the backward reduce-scatter is quantized to
// INT8 or INT4 (qgZ).  Format (the same as the CPU oracle's): blocks of 256
// elements from the start of the buffer or bucket; per block lo = min,
// hi = max (NaN propagates), scale = (hi - lo) / (2^bits - 1), code =
// rint((x - lo) / scale) clamped to [0, 2^bits - 1] (0 when scale is 0, 0
// for a NaN), the subtraction and the division each rounded once;
// dequantized x' = lo + code * scale.
//
// Two exact bit-level shortcuts keep the per-element cost to a few adds:
// for 0 <= u < 2^22, u + 2^23 (rounded to nearest even) holds rint(u) in its
// low mantissa bits; and the float with bits 0x4B000000 | q, minus 2^23, is
// exactly q for any q < 2^23.  Neither changes a result.  Codes: one byte each (INT8), or two
// per byte (INT4, even element in the low nibble).  Scales: {scale, lo}
// float pairs, one per block.
//
// One warp owns one 256-element block at a time (8 elements per lane), two
// or four blocks per iteration so that their loads are in flight together: the
// block's min and max are one warp reduction each (redux.sync); codes leave as 8-byte (INT8) or
// 4-byte (INT4) stores per lane.  All kernels are HBM streams.

#include "zero_device.cuh"

namespace zg {
namespace {

// min/max that return NaN when either input is NaN (one instruction each),
// and their warp-wide forms.
__device__ __forceinline__ float qmin(float a, float b) {
    float d;
    asm("min.NaN.f32 %0, %1, %2;" : "=f"(d) : "f"(a), "f"(b));
    return d;
}
__device__ __forceinline__ float qmax(float a, float b) {
    float d;
    asm("max.NaN.f32 %0, %1, %2;" : "=f"(d) : "f"(a), "f"(b));
    return d;
}
__device__ __forceinline__ float warp_qmin(float a) {
    float d;
    asm volatile("redux.sync.min.NaN.f32 %0, %1, 0xffffffff;" : "=f"(d) : "f"(a));
    return d;
}
__device__ __forceinline__ float warp_qmax(float a) {
    float d;
    asm volatile("redux.sync.max.NaN.f32 %0, %1, 0xffffffff;" : "=f"(d) : "f"(a));
    return d;
}

constexpr float kTwo23 = 8388608.0f;

// 1/x from the hardware's approximate reciprocal (1 ulp); used only by the
// screen in codes8, whose margin allows 2^-22 relative.
__device__ __forceinline__ float rcp_approx(float x) {
    float r;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
}

// Two fp32 lanes in one 64-bit register for the packed add/sub/mul.rn.f32x2
// of sm_100 and later: each half is an ordinary fp32 operation rounded once,
// so results are those of the scalar instructions, at half the issue cost.
using f2 = unsigned long long;
__device__ __forceinline__ f2 f2pack(float a, float b) {
    f2 r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
    return r;
}
__device__ __forceinline__ f2 f2bits(uint32_t a, uint32_t b) {
    f2 r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "r"(a), "r"(b));
    return r;
}
__device__ __forceinline__ void f2unpack(f2 x, float& a, float& b) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(x));
}
__device__ __forceinline__ f2 f2add(f2 a, f2 b) {
    f2 r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ f2 f2sub(f2 a, f2 b) {
    f2 r;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ f2 f2mul(f2 a, f2 b) {
    f2 r;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}

// A lane's codes rint(clamp(q, 0, top)) for q = (x - lo) / scale rounded once
// (IEEE division), a NaN q giving 0 (fmaxf returns the other operand), as
// the words tb[k] = bits of 2^23 + code: the code is tb[k] & 0x1FF, and its
// low byte for INT8.  Only elements k < nv are meaningful; finish_codes
// forms the codes (0 for absent elements and when scale is 0).
//
// The division is taken only where it can matter.  Let d = x - lo (rounded
// once) and rcp = 1/scale to within 2^-22 relative (the hardware's
// approximate reciprocal, which the PTX ISA documents to 1 ulp, 2^-23).  The
// exact product p = d * rcp lies within 2^-22 p of d / scale, its rounding u
// within 2^-24 u of p, and the rounded quotient Q within 2^-24 Q of
// d / scale; with d / scale < 256, Q lies within 2^-14 + 2^-15 < 2^-13 of
// u.  The code is read from u + 2^23 (for 0 <= u < 2^22 its low mantissa
// bits hold k = rint(u); k = rint(p) should the compiler fuse the multiply
// into the add, which changes nothing below), and r = u - ((u + 2^23) -
// 2^23) = u - k is exact.  When |r| < 0.5 - 2^-12, |Q - k| < 0.5 - 2^-12 +
// 2^-13 < 0.5, so k = rint(Q): the code.  Otherwise the lane divides all its
// elements again: for values spread over the levels that is one lane in
// about 250.
//
// No clamp is needed on the screened path.  It runs only for a block of
// finite values whose scale is a normal number in [2^-100, 2^100] (`fast`;
// the bounds above assume no underflow or overflow), and there every
// present x >= lo, so 0 <= d <= hi - lo and 0 <= Q, u < top + 2^-12: k lies
// in [0, top], and rint(clamp(Q)) = rint(Q) (Q > top only by less than 0.5).
// Absent elements (index >= nv: copies of a present one, or 0 in a lane
// with none) may only add a division: their codes are forced to 0, and a
// NaN r of theirs drops out of the fmaxf.  A
// block that is not fast (NaN, infinite, zero or extreme range) divides
// every element with the clamp.
__device__ __forceinline__ void codes8(const float (&x)[8], float lo, float scale, float rcp, bool fast, float top,
                                       uint32_t (&tb)[8]) {
    float t[8];
    float rmax = 0.0f;
    // pairs of elements in packed operations (each half one IEEE-rounded
    // fp32 operation)
    const f2 lo2 = f2pack(lo, lo), rcp2 = f2pack(rcp, rcp), two23 = f2pack(kTwo23, kTwo23);
#pragma unroll
    for (int k = 0; k < 8; k += 2) {
        float r0, r1;
        const f2 u = f2mul(f2sub(f2pack(x[k], x[k + 1]), lo2), rcp2);
        const f2 tt = f2add(u, two23);
        f2unpack(f2sub(u, f2sub(tt, two23)), r0, r1);
        f2unpack(tt, t[k], t[k + 1]);
        rmax = fmaxf(rmax, fmaxf(fabsf(r0), fabsf(r1)));
    }
    // 0.5 - 2^-12
    if (!fast || !(rmax < 0x1.ffcp-2f)) {
#pragma unroll
        for (int k = 0; k < 8; ++k)
            t[k] = __fadd_rn(fminf(fmaxf(__fdiv_rn(__fsub_rn(x[k], lo), scale), 0.0f), top), kTwo23);
    }
#pragma unroll
    for (int k = 0; k < 8; ++k) tb[k] = __float_as_uint(t[k]);
}

// The codes of a lane from codes8's words.
__device__ __forceinline__ void finish_codes(const uint32_t (&tb)[8], int nv, float scale, uint32_t (&q)[8]) {
#pragma unroll
    for (int k = 0; k < 8; ++k) q[k] = (k < nv && scale != 0.0f) ? (tb[k] & 0x1FFu) : 0u;
}

// float(q) for q < 2^23, exactly.
__device__ __forceinline__ float as_float(uint32_t q) {
    return __fsub_rn(__uint_as_float(0x4B000000u | q), kTwo23);
}

__device__ __forceinline__ float dequant(uint32_t q, float scale, float lo) {
    return __fadd_rn(lo, __fmul_rn(as_float(q), scale));
}

// Lane's 8 values of a block of a 16-bit buffer (elements >= count are absent).
template <int DT>
__device__ __forceinline__ int load_lane8(const void* src, uint64_t e0, uint64_t count, bool vec, float (&x)[8]) {
    const int nv = e0 >= count ? 0 : static_cast<int>(count - e0 < 8 ? count - e0 : 8);
    if (vec && nv == 8) {
        uint32_t raw[8];
        Io8s16::ld16(src, e0, raw);
#pragma unroll
        for (int k = 0; k < 8; ++k) x[k] = widen<DT>(raw[k]);
    } else {
        // absent elements repeat the lane's first one (0 in a lane with none),
        // so that they change no min or max
        const unsigned short* s = reinterpret_cast<const unsigned short*>(src);
        const float x0 = nv > 0 ? widen<DT>(s[e0]) : 0.0f;
#pragma unroll
        for (int k = 0; k < 8; ++k) x[k] = (k < nv) ? widen<DT>(s[e0 + k]) : x0;
    }
    return nv;
}

// Block min/max over the warp; every lane gets {scale, lo}, the
// approximate reciprocal of the scale and whether codes8 may screen with it.
template <int BITS>
__device__ __forceinline__ void block_scale(const float (&x)[8], int nv, float& scale, float& lo, float& rcp,
                                            bool& fast) {
    // absent elements repeat a present one (load_lane8); a lane with none
    // contributes the identities
    float mn = x[0], mx = x[0];
#pragma unroll
    for (int k = 1; k < 8; ++k) {
        mn = qmin(mn, x[k]);
        mx = qmax(mx, x[k]);
    }
    if (nv == 0) {
        mn = __int_as_float(0x7F800000);
        mx = -__int_as_float(0x7F800000);
    }
    // warp-wide, then +0.0 makes a zero bound +0 whatever the order of ties
    mn = __fadd_rn(warp_qmin(mn), 0.0f);
    mx = __fadd_rn(warp_qmax(mx), 0.0f);
    lo = mn;
    const float range = __fsub_rn(mx, mn);
    const float top = static_cast<float>((1 << BITS) - 1);
    scale = __fdiv_rn(range, top);
    fast = scale >= 0x1p-100f && scale <= 0x1p100f;
    rcp = fast ? rcp_approx(scale) : 0.0f;
}

// The low bytes of eight words (codes, or codes8's words for INT8) packed
// little-endian into 8 bytes.
__device__ __forceinline__ uint2 pack_u8x8(const uint32_t (&q)[8]) {
    uint2 w;
    w.x = __byte_perm(__byte_perm(q[0], q[1], 0x0040u), __byte_perm(q[2], q[3], 0x0040u), 0x5410u);
    w.y = __byte_perm(__byte_perm(q[4], q[5], 0x0040u), __byte_perm(q[6], q[7], 0x0040u), 0x5410u);
    return w;
}

// Store a lane's 8 codes at element e0 of a code buffer.
template <int BITS>
__device__ __forceinline__ void store_codes(void* codes, uint64_t e0, int nv, const uint32_t (&q)[8]) {
    if (BITS == 8) {
        unsigned char* c = static_cast<unsigned char*>(codes) + e0;
        if (nv == 8) {
            __stcs(reinterpret_cast<uint2*>(c), pack_u8x8(q));
        } else {
            for (int k = 0; k < nv; ++k) c[k] = static_cast<unsigned char>(q[k]);
        }
    } else {
        unsigned char* c = static_cast<unsigned char*>(codes) + (e0 >> 1);
        if (nv == 8) {
            const uint32_t w = q[0] | (q[1] << 4) | (q[2] << 8) | (q[3] << 12) | (q[4] << 16) | (q[5] << 20) |
                               (q[6] << 24) | (q[7] << 28);
            __stcs(reinterpret_cast<unsigned int*>(c), w);
        } else {
            for (int k = 0; k < nv; k += 2) {
                const uint32_t hi = (k + 1 < nv) ? q[k + 1] : 0u;
                c[k >> 1] = static_cast<unsigned char>(q[k] | (hi << 4));
            }
        }
    }
}

// A lane's 8 codes at element e0 (e0 % 8 == 0).
template <int BITS>
__device__ __forceinline__ void load_codes8(const void* codes, uint64_t e0, uint32_t (&q)[8]) {
    if (BITS == 8) {
        const uint2 w = __ldcs(reinterpret_cast<const uint2*>(static_cast<const unsigned char*>(codes) + e0));
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            q[k] = (w.x >> (8 * k)) & 0xFFu;
            q[4 + k] = (w.y >> (8 * k)) & 0xFFu;
        }
    } else {
        const uint32_t w = __ldcs(reinterpret_cast<const unsigned int*>(static_cast<const unsigned char*>(codes) + (e0 >> 1)));
#pragma unroll
        for (int k = 0; k < 8; ++k) q[k] = (w >> (4 * k)) & 0xFu;
    }
}

// lo + q*scale for a pair, with the multiply packed and the add scalar: a
// packed multiply feeding a packed add may be fused into one packed FMA
// (observed: results then differ from two separately rounded operations).
__device__ __forceinline__ f2 f2dequant(f2 q_biased, f2 two23, f2 sc, float lo) {
    f2 prod;
    asm("{\n\t.reg .b64 t;\n\tsub.rn.f32x2 t, %1, %2;\n\tmul.rn.f32x2 %0, t, %3;\n\t}"
        : "=l"(prod) : "l"(q_biased), "l"(two23), "l"(sc));
    float p0, p1;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(p0), "=f"(p1) : "l"(prod));
    return f2pack(__fadd_rn(lo, p0), __fadd_rn(lo, p1));
}


// A lane's 8 codes at element e0 as they lie in memory: 8 bytes (INT8,
// both words used) or 4 bytes (INT4, .y unused).
template <int BITS>
__device__ __forceinline__ uint2 load_codes8_raw(const void* codes, uint64_t e0) {
    if (BITS == 8) return __ldcs(reinterpret_cast<const uint2*>(static_cast<const unsigned char*>(codes) + e0));
    return make_uint2(__ldcs(reinterpret_cast<const unsigned int*>(static_cast<const unsigned char*>(codes) + (e0 >> 1))), 0u);
}

// Those codes as four pairs of 2^23-biased floats (0x4B000000 | code):
// subtracting 2^23 gives the codes exactly.  Kept apart from the load so
// that the loads of several ranks hold only their raw words in registers.
template <int BITS>
__device__ __forceinline__ void expand_codes8(uint2 w, f2 (&q)[4]) {
    if (BITS == 8) {
        q[0] = f2bits(__byte_perm(w.x, 0x4B000000u, 0x7540u), __byte_perm(w.x, 0x4B000000u, 0x7541u));
        q[1] = f2bits(__byte_perm(w.x, 0x4B000000u, 0x7542u), __byte_perm(w.x, 0x4B000000u, 0x7543u));
        q[2] = f2bits(__byte_perm(w.y, 0x4B000000u, 0x7540u), __byte_perm(w.y, 0x4B000000u, 0x7541u));
        q[3] = f2bits(__byte_perm(w.y, 0x4B000000u, 0x7542u), __byte_perm(w.y, 0x4B000000u, 0x7543u));
    } else {
        // even elements are the low nibbles, odd ones the high nibbles: split
        // them into bytes, then place each byte under the 2^23 exponent
        const uint32_t ev = w.x & 0x0F0F0F0Fu, od = (w.x >> 4) & 0x0F0F0F0Fu;
        q[0] = f2bits(__byte_perm(ev, 0x4B000000u, 0x7540u), __byte_perm(od, 0x4B000000u, 0x7540u));
        q[1] = f2bits(__byte_perm(ev, 0x4B000000u, 0x7541u), __byte_perm(od, 0x4B000000u, 0x7541u));
        q[2] = f2bits(__byte_perm(ev, 0x4B000000u, 0x7542u), __byte_perm(od, 0x4B000000u, 0x7542u));
        q[3] = f2bits(__byte_perm(ev, 0x4B000000u, 0x7543u), __byte_perm(od, 0x4B000000u, 0x7543u));
    }
}

template <int BITS>
__device__ __forceinline__ uint32_t load_code1(const void* codes, uint64_t e) {
    if (BITS == 8) return static_cast<const unsigned char*>(codes)[e];
    const uint32_t b = static_cast<const unsigned char*>(codes)[e >> 1];
    return (e & 1) ? (b >> 4) : (b & 0xFu);
}

__device__ __forceinline__ uint64_t warp_id() { return (static_cast<uint64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5; }
__device__ __forceinline__ uint64_t warp_count() { return (static_cast<uint64_t>(gridDim.x) * blockDim.x) >> 5; }

// Warp-iterations per chunk for the quantized gather: as few as leave a
// launch about q_chunk_target(N) chunks, at most 4.  With N = 8 the finest
// chunks measured best (no partials to commit): at ψ = 2^29, 2e8-element
// buckets, a step's gathers took 1.4 % less than with 2048 chunks per
// launch, and the step 1.1 % less than with 8192.  With few ranks a chunk
// writes few bytes and its closing barrier weighs more: at N = 2 the same
// step took 3.61 ms with 8192 chunks per launch (4 iterations each) against
// 3.69 ms with 32768, and at N = 4 the step's gathers 1.297 against 1.312 ms.
constexpr int kQSmallN = 4;
__host__ __device__ inline uint64_t q_chunk_target(int n_ranks) { return n_ranks <= kQSmallN ? 8192 : 32768; }
__host__ __device__ inline int q_chunk_u(uint64_t iters, int n_ranks) {
    const uint64_t u = iters / q_chunk_target(n_ranks);
    return u >= 4 ? 4 : (u < 1 ? 1 : static_cast<int>(u));
}

// ------------------------------------------------------------------ kernels
// Blocks per warp iteration (their loads are in flight together): two for
// the gather, whose stores to N ranks dominate; four for the one-output
// quantize, which is read-bound.
constexpr int kQUnrollGather = 2;
constexpr int kQUnrollQuant = 4;

// Quantize U consecutive blocks starting at block blk0 of src (count
// elements) and hand each block's lane words (codes8) and {scale, lo} to
// `emit`.
template <int DT, int BITS, int kQUnroll, class Emit>
__device__ __forceinline__ void quantize_blocks_u(const unsigned short* src, uint64_t count, uint64_t blk0,
                                                  uint64_t nb, bool vec, int lane, Emit&& emit) {
    const float top = static_cast<float>((1 << BITS) - 1);
    float x[kQUnroll][8];
    int nv[kQUnroll];
#pragma unroll
    for (int u = 0; u < kQUnroll; ++u) {
        const uint64_t e0 = (blk0 + u) * kQBlock + static_cast<uint64_t>(lane) * 8;
        nv[u] = (blk0 + u < nb) ? load_lane8<DT>(src, e0, count, vec, x[u]) : 0;
    }
#pragma unroll
    for (int u = 0; u < kQUnroll; ++u) {
        if (blk0 + u >= nb) break;
        float scale, lo, rcp;
        bool fast;
        block_scale<BITS>(x[u], nv[u], scale, lo, rcp, fast);
        uint32_t tb[8];
        codes8(x[u], lo, scale, rcp, fast, top, tb);
        emit(blk0 + u, (blk0 + u) * kQBlock + static_cast<uint64_t>(lane) * 8, nv[u], tb, scale, lo);
    }
}

// One 16-bit buffer (grads[0] + base, count elements) -> codes (params[0])
// and {scale, lo} pairs (qdst[0]).
template <int DT, int BITS>
__global__ void __launch_bounds__(kThreads) k_quantize(const __grid_constant__ Args a) {
    pdl_enter();
    const int lane = threadIdx.x & 31;
    const uint64_t nb = (a.count + kQBlock - 1) / kQBlock;
    const unsigned short* src = static_cast<const unsigned short*>(a.grads[0]) + a.base;
    for (uint64_t blk0 = warp_id() * kQUnrollQuant; blk0 < nb; blk0 += warp_count() * kQUnrollQuant) {
        quantize_blocks_u<DT, BITS, kQUnrollQuant>(src, a.count, blk0, nb, a.qvec != 0, lane,
                                    [&](uint64_t blk, uint64_t e0, int nv, const uint32_t (&tb)[8], float scale,
                                        float lo) {
                                        uint32_t q[8];
                                        finish_codes(tb, nv, scale, q);
                                        if (nv > 0) store_codes<BITS>(a.params[0], e0, nv, q);
                                        if (lane == 0)
                                            *reinterpret_cast<float2*>(a.qdst[0] + 2 * blk) = make_float2(scale, lo);
                                    });
    }
}

// ZeRO-3 quantized gather (qwZ): bucket [base, base+count) of the 16-bit
// shard (grads[0]) -> for every rank r: codes (params[r]) and scales (qdst[r]).
// Chunked like the other persistent kernels (zero_device.cuh): a chunk is
// U iterations of the CTA's 8 warps, kQUnrollGather blocks per warp each.
// Six CTAs per SM (40 registers, no spill): the quantizing arithmetic wants
// the extra warps; four per SM (56 registers) measured 2 % slower at N = 8
// and 6 % at N = 2, and fewer per SM slower still.
template <int DT>
__global__ void __launch_bounds__(kThreads, 6) k_gather_q8(const __grid_constant__ Args a) {
    pdl_enter();
    __shared__ unsigned long long s_c[2];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const uint64_t nb = (a.count + kQBlock - 1) / kQBlock;
    const unsigned short* src = static_cast<const unsigned short*>(a.grads[0]) + a.base;
    // one "vector" = one warp-iteration's blocks; kThreads vectors per U unit
    // would be too coarse here, so the chunk length counts warp-iterations
    constexpr uint64_t kPerIter = static_cast<uint64_t>(kThreads / 32) * kQUnrollGather;
    const uint64_t iters = (nb + kPerIter - 1) / kPerIter;
    const int U = q_chunk_u(iters, a.n_ranks);
    const uint64_t nchunks = (iters + U - 1) / U;
    ChunkCtr* ctr = a.ws.ctrs + a.ctr_slot;
    Chunks ch(ctr, s_c, nchunks);
    for (;;) {
      const uint64_t c = ch.current();
      if (c >= nchunks) break;
      ch.prefetch();
      for (int u = 0; u < U; ++u) {
        const uint64_t blk0 = (c * U + u) * kPerIter + static_cast<uint64_t>(warp) * kQUnrollGather;
        if (blk0 >= nb) break;
        quantize_blocks_u<DT, 8, kQUnrollGather>(src, a.count, blk0, nb, a.qvec != 0, lane,
                                 [&](uint64_t blk, uint64_t e0, int nv, const uint32_t (&tb)[8], float scale,
                                     float lo) {
                                     // the same 8 bytes to every rank, packed once, straight
                                     // from the words' low bytes (all 0 when scale is 0)
                                     if (nv == 8) {
                                         uint2 w = pack_u8x8(tb);
                                         if (scale == 0.0f) w = make_uint2(0u, 0u);
                                         for (int r = 0; r < a.n_ranks; ++r)
                                             __stcs(reinterpret_cast<uint2*>(static_cast<unsigned char*>(a.params[r]) + e0), w);
                                     } else if (nv > 0) {
                                         uint32_t q[8];
                                         finish_codes(tb, nv, scale, q);
                                         for (int r = 0; r < a.n_ranks; ++r) store_codes<8>(a.params[r], e0, nv, q);
                                     }
                                     // lane r writes rank r's {scale, lo}
                                     for (int r = lane; r < a.n_ranks; r += 32)
                                         *reinterpret_cast<float2*>(a.qdst[r] + 2 * blk) = make_float2(scale, lo);
                                 });
      }
      __syncthreads();
      ch.advance();
    }
}

// codes (grads[0]) + scales (qsrc[0]) -> 16-bit buffer (params[0]), count elements.
template <int DT, int BITS>
__global__ void __launch_bounds__(kThreads) k_dequantize(const __grid_constant__ Args a) {
    pdl_enter();
    const uint64_t nv8 = (a.count + 7) / 8;
    for (uint64_t t = thread_id(); t < nv8; t += grid_threads()) {
        const uint64_t e0 = t * 8;
        const uint64_t blk = e0 / kQBlock;
        const float scale = a.qsrc[0][2 * blk], lo = a.qsrc[0][2 * blk + 1];
        const int nv = static_cast<int>(a.count - e0 < 8 ? a.count - e0 : 8);
        uint32_t out[8];
        if (nv == 8) {
            uint32_t q[8];
            load_codes8<BITS>(a.grads[0], e0, q);
#pragma unroll
            for (int k = 0; k < 8; ++k) out[k] = narrow<DT>(dequant(q[k], scale, lo));
            Io8s16::st16(a.params[0], e0, out);
        } else {
            for (int k = 0; k < nv; ++k)
                reinterpret_cast<unsigned short*>(a.params[0])[e0 + k] =
                    static_cast<unsigned short>(narrow<DT>(dequant(load_code1<BITS>(a.grads[0], e0 + k), scale, lo)));
        }
    }
}

// Sum over ranks (order 0..N-1, from +0) of the dequantized gradients of W
// elements at bucket-local index j, then unscale: s += lo + q*scale per
// rank, each operation rounded once.  Ranks go in chunks of 8 whose code and
// scale loads are all issued before any arithmetic; the 8-wide path works on
// packed pairs.
template <int BITS, int W>
__device__ __forceinline__ void reduce_group_q(const Args& a, uint64_t j, const Pro& pro, float (&g)[W]) {
    const uint64_t blk = j / kQBlock;
    const int n = a.n_ranks;
    if (W == 8) {
        const f2 two23 = f2pack(kTwo23, kTwo23);
        f2 s2[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) s2[k] = f2pack(0.0f, 0.0f);
        int r = 0;
        for (; r + 8 <= n; r += 8) {
            uint2 w[8];
            float2 sl[8];
#pragma unroll
            for (int t = 0; t < 8; ++t) {
                sl[t] = *reinterpret_cast<const float2*>(a.qsrc[r + t] + 2 * blk);
                w[t] = load_codes8_raw<BITS>(a.grads[r + t], j);
            }
#pragma unroll
            for (int t = 0; t < 8; ++t) {
                f2 q[4];
                expand_codes8<BITS>(w[t], q);
                const f2 sc = f2pack(sl[t].x, sl[t].x);
#pragma unroll
                for (int k = 0; k < 4; ++k) s2[k] = f2add(s2[k], f2dequant(q[k], two23, sc, sl[t].y));
            }
        }
        for (; r < n; ++r) {
            const float2 sl = *reinterpret_cast<const float2*>(a.qsrc[r] + 2 * blk);
            f2 q[4];
            expand_codes8<BITS>(load_codes8_raw<BITS>(a.grads[r], j), q);
            const f2 sc = f2pack(sl.x, sl.x);
#pragma unroll
            for (int k = 0; k < 4; ++k) s2[k] = f2add(s2[k], f2dequant(q[k], two23, sc, sl.y));
        }
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            float x0, x1;
            f2unpack(s2[k], x0, x1);
            g[2 * k] = pro.use_div ? __fdiv_rn(x0, pro.den) : __fmul_rn(x0, pro.inv);
            g[2 * k + 1] = pro.use_div ? __fdiv_rn(x1, pro.den) : __fmul_rn(x1, pro.inv);
        }
    } else {
        float s[W];
#pragma unroll
        for (int k = 0; k < W; ++k) s[k] = 0.0f;
        for (int r = 0; r < n; ++r) {
            const float2 sl = *reinterpret_cast<const float2*>(a.qsrc[r] + 2 * blk);
#pragma unroll
            for (int k = 0; k < W; ++k) s[k] = __fadd_rn(s[k], dequant(load_code1<BITS>(a.grads[r], j + k), sl.x, sl.y));
        }
#pragma unroll
        for (int k = 0; k < W; ++k) g[k] = pro.use_div ? __fdiv_rn(s[k], pro.den) : __fmul_rn(s[k], pro.inv);
    }
}

// ZeRO-3 reduce-scatter of bucket [base, base+count) from the N ranks'
// quantized gradients (qgZ): as k_rs, with the ranks' values dequantized.
// Static grid-stride: this kernel waits on its loads, and chunked
// scheduling's block barriers cost more (+6 % for int8, measured at 3 CTAs
// per SM) than the balance gains.  4 CTAs per SM (64 registers, a short
// spill): against 3, the int4 form's reduce-scatters took 3.9 % less, and
// the int8 form's (since its codes stay raw words until used) 4.9 / 4.2 /
// 0.7 % less at N = 2 / 4 / 8 (ψ = 2^29).
template <int DT, class IO, int BITS, bool SPEC>
__global__ void __launch_bounds__(kThreads, 4) k_rs_q(const __grid_constant__ Args a) {
    pdl_enter();
    constexpr int W = IO::W;
    __shared__ Pro pro;
    prologue_reduce(a, pro, SPEC);
    const uint64_t src = static_cast<uint64_t>(pro.live) * a.slot_stride;
    const uint64_t dst = static_cast<uint64_t>(pro.live ^ 1) * a.slot_stride;
    const uint64_t nvec = a.count / W;
    double acc = 0.0;
    int bad = 0;
    for (uint64_t vi = thread_id(); vi < nvec; vi += grid_threads()) {
        const uint64_t j = vi * W;
        const uint64_t gi = a.base + j;
        float g[W];
        reduce_group_q<BITS, W>(a, j, pro, g);
        const int valid = valid_count(gi, W, a.psi);
        norm_group<W>(g, valid, acc, bad);
        if (SPEC) {
            float p[W], m[W], v[W];
            IO::ldf(a.master + src, gi, p);
            IO::ldf(a.m + src, gi, m);
            IO::ldf(a.v + src, gi, v);
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
            IO::st16(a.params[0], gi, q);
        } else {
#pragma unroll
            for (int k = 0; k < W; ++k)
                if (k >= valid) g[k] = 0.0f;
            IO::stf(a.ws.ghat, gi, g);
        }
    }
    const double blk = block_sum(acc);
    const int flag = __syncthreads_or(bad);
    if (publish(a, blk, flag, a.ws.partials, a.ws.flags)) {
        double qsum;
        int f;
        gather_partials(a.ws.partials, a.ws.flags, gridDim.x, qsum, f);
        if (threadIdx.x == 0) {
            a.ws.bucket_norm[a.bucket_index] = qsum;
            a.ws.bucket_flag[a.bucket_index] = f;
            a.ws.status->ticket = 0u;
        }
    }
}

template <int DT, int BITS>
cudaError_t launch_db(QKind kind, Vec vec, const Args& a, cudaStream_t s) {
    const uint64_t nb = (a.count + kQBlock - 1) / kQBlock;
    switch (kind) {
        case QKind::kQuantize:
            return run(k_quantize<DT, BITS>, a, (nb + kQUnrollQuant - 1) / kQUnrollQuant * 32, s, nullptr);
        case QKind::kGatherQ8: {
            // one CTA per chunk at most (run() sizes the grid from threads)
            const uint64_t per_iter = static_cast<uint64_t>(kThreads / 32) * kQUnrollGather;
            const uint64_t iters = (nb + per_iter - 1) / per_iter;
            const uint64_t nch = (iters + q_chunk_u(iters, a.n_ranks) - 1) / q_chunk_u(iters, a.n_ranks);
            return run(k_gather_q8<DT>, a, nch * kThreads, s, nullptr);
        }
        case QKind::kDequantize: return run(k_dequantize<DT, BITS>, a, (a.count + 7) / 8, s, nullptr);
        case QKind::kRsQSpec:
        case QKind::kRsQWs: {
            const bool spec = kind == QKind::kRsQSpec;
            switch (vec) {
                case Vec::k8s32:
                    return spec ? run(k_rs_q<DT, Io8s32, BITS, true>, a, a.count / 8, s, nullptr)
                                : run(k_rs_q<DT, Io8s32, BITS, false>, a, a.count / 8, s, nullptr);
                case Vec::k8s16:
                    return spec ? run(k_rs_q<DT, Io8s16, BITS, true>, a, a.count / 8, s, nullptr)
                                : run(k_rs_q<DT, Io8s16, BITS, false>, a, a.count / 8, s, nullptr);
                default:
                    return spec ? run(k_rs_q<DT, Io1, BITS, true>, a, a.count, s, nullptr)
                                : run(k_rs_q<DT, Io1, BITS, false>, a, a.count, s, nullptr);
            }
        }
    }
    return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_q(QKind kind, int dtype, int bits, Vec vec, const Args& a, cudaStream_t s) {
    if (dtype == kFp16) return bits == 8 ? launch_db<kFp16, 8>(kind, vec, a, s) : launch_db<kFp16, 4>(kind, vec, a, s);
    return bits == 8 ? launch_db<kBf16, 8>(kind, vec, a, s) : launch_db<kBf16, 4>(kind, vec, a, s);
}

}  // namespace zg
