// Device building blocks of the single-pass scan: operators, status words of
// the decoupled look-back, tile loads/stores, and the thread/warp/block scan.
//
// Scan definitions (inclusive y[i] = x[0] (+) ... (+) x[i]; exclusive y[0] = I,
// y[i] = x[0] (+) ... (+) x[i-1]) follow "Lecture 7: Parallel pattern -- prefix
// sum / scan" (UIUC ECE408 notes), section 1, and "Chapter 9 Parallel Patterns:
// Prefix Sum - Scan Algorithms" (PMPP notes), section 9.1.
#pragma once
#include <cstdint>
#include <type_traits>
#include <cuda_runtime.h>

#include "sc_params.h"

namespace scg {

// ----------------------------------------------------------------- operators
// Each operator has an element type T (what the tile is scanned in) and a
// carry type C (what travels between tiles through the look-back).  Only the
// float32 sum has C != T: its inter-tile carry is a float-float pair so that
// the error of a prefix stays a small multiple of eps * sum|x| however many
// tiles precede it.

struct OpSumU32 {  // int32 and uint32 sums: two's-complement wraparound mod 2^32
    using T = uint32_t;
    using C = uint32_t;
    __device__ __forceinline__ static T identity() { return 0u; }
    __device__ __forceinline__ static T op(T a, T b) { return a + b; }
    __device__ __forceinline__ static C c_identity() { return 0u; }
    __device__ __forceinline__ static C c_op(C a, C b) { return a + b; }
    __device__ __forceinline__ static C lift(T a) { return a; }
    __device__ __forceinline__ static T lower(C c) { return c; }
};

// Sum of two float-float numbers (x = high part, y = low part, |y| <= ulp(x)/2):
// Knuth's error-free TwoSum of the high parts, the low parts added to its
// error, then a fast renormalisation (Dekker).  Relative error about 2^-44 of
// |a| + |b|; float32 operations only.
__device__ __forceinline__ float2 ff_add(float2 a, float2 b) {
    const float s = __fadd_rn(a.x, b.x);
    if (!isfinite(s)) return make_float2(s, 0.0f);  // inf or NaN, as a float32 sum gives it; no low part
    const float bv = __fsub_rn(s, a.x);
    const float e = __fadd_rn(__fsub_rn(a.x, __fsub_rn(s, bv)), __fsub_rn(b.x, bv));  // a.x + b.x == s + e exactly
    const float lo = __fadd_rn(e, __fadd_rn(a.y, b.y));
    const float hi = __fadd_rn(s, lo);
    return make_float2(hi, __fsub_rn(lo, __fsub_rn(hi, s)));
}

// float32 sums: each tile in float32; the carry between tiles as a float-float
// pair, so that a prefix chained through many tiles keeps about 44 bits
// (GB300's float64 units are slow enough that a float64 carry cost 7-8 % of
// the scan's time).
struct OpSumF32 {
    using T = float;
    using C = float2;
    __device__ __forceinline__ static T identity() { return 0.0f; }
    __device__ __forceinline__ static T op(T a, T b) { return __fadd_rn(a, b); }
    __device__ __forceinline__ static C c_identity() { return make_float2(0.0f, 0.0f); }
    __device__ __forceinline__ static C c_op(C a, C b) { return ff_add(a, b); }
    __device__ __forceinline__ static C lift(T a) { return make_float2(a, 0.0f); }
    __device__ __forceinline__ static T lower(C c) { return __fadd_rn(c.x, c.y); }
    // look-back: aggregates folded in float32, one float-float add onto the prefix
    static constexpr bool kLowFold = true;
    using L = float;
    __device__ __forceinline__ static L low(C c) { return c.x; }
    __device__ __forceinline__ static L low_identity() { return 0.0f; }
    __device__ __forceinline__ static L low_op(L a, L b) { return __fadd_rn(a, b); }
    __device__ __forceinline__ static C with_low(C prefix, L s) { return ff_add(prefix, make_float2(s, 0.0f)); }
};

struct OpMaxI32 {  // identity INT32_MIN (the "-infinity" of the PMPP identity table)
    using T = int32_t;
    using C = int32_t;
    __device__ __forceinline__ static T identity() { return INT32_MIN; }
    __device__ __forceinline__ static T op(T a, T b) { return max(a, b); }
    __device__ __forceinline__ static C c_identity() { return INT32_MIN; }
    __device__ __forceinline__ static C c_op(C a, C b) { return max(a, b); }
    __device__ __forceinline__ static C lift(T a) { return a; }
    __device__ __forceinline__ static T lower(C c) { return c; }
};

// Affine maps h -> a*h + b (mod 2^32) stored as uint2 {x = a, y = b}.
// l (+) r applies l first, then r:  (r.a*l.a, r.a*l.b + r.b).  Not commutative,
// so every combine below keeps the earlier operand on the left.
struct OpAffineU32 {
    using T = uint2;
    using C = uint2;
    __device__ __forceinline__ static T identity() { return make_uint2(1u, 0u); }
    __device__ __forceinline__ static T op(T l, T r) { return make_uint2(r.x * l.x, r.x * l.y + r.y); }
    __device__ __forceinline__ static C c_identity() { return make_uint2(1u, 0u); }
    __device__ __forceinline__ static C c_op(C l, C r) { return op(l, r); }
    __device__ __forceinline__ static C lift(T a) { return a; }
    __device__ __forceinline__ static T lower(C c) { return c; }
};

// ---- more operators ("Lecture 7" notes, section 1, operator list; PMPP
// notes, section 9.1, identity table).  Integer operators act on the
// unsigned bits (wraparound); max/min compare in the value's own type.

// Identity-preserving helpers for the generic operators below.
template <class V> struct Extremes;
template <> struct Extremes<int32_t> {
    __device__ __forceinline__ static int32_t lowest() { return INT32_MIN; }
    __device__ __forceinline__ static int32_t highest() { return INT32_MAX; }
};
template <> struct Extremes<uint32_t> {
    __device__ __forceinline__ static uint32_t lowest() { return 0u; }
    __device__ __forceinline__ static uint32_t highest() { return 0xffffffffu; }
};
template <> struct Extremes<long long> {
    __device__ __forceinline__ static long long lowest() { return (long long)0x8000000000000000ull; }
    __device__ __forceinline__ static long long highest() { return 0x7fffffffffffffffll; }
};
template <> struct Extremes<unsigned long long> {
    __device__ __forceinline__ static unsigned long long lowest() { return 0ull; }
    __device__ __forceinline__ static unsigned long long highest() { return ~0ull; }
};
template <> struct Extremes<float> {
    __device__ __forceinline__ static float lowest() { return __int_as_float(0xff800000); }   // -inf
    __device__ __forceinline__ static float highest() { return __int_as_float(0x7f800000); }  // +inf
};
template <> struct Extremes<double> {
    __device__ __forceinline__ static double lowest() { return __longlong_as_double((long long)0xfff0000000000000ull); }
    __device__ __forceinline__ static double highest() { return __longlong_as_double(0x7ff0000000000000ll); }
};

// Operators whose combine costs several instructions (or slow float64 units)
// declare kHeavyCombine = true; kernels may then trade shared memory for
// fewer combines per element.
template <class Op, class = void>
struct HeavyCombine { static constexpr bool value = false; };
template <class Op>
struct HeavyCombine<Op, std::void_t<decltype(Op::kHeavyCombine)>> { static constexpr bool value = Op::kHeavyCombine; };

// An operator whose carry has the element's type.
template <class V, class Self>
struct SameCarry {
    using T = V;
    using C = V;
    __device__ __forceinline__ static C c_identity() { return Self::identity(); }
    __device__ __forceinline__ static C c_op(C a, C b) { return Self::op(a, b); }
    __device__ __forceinline__ static C lift(T a) { return a; }
    __device__ __forceinline__ static T lower(C c) { return c; }
};

template <class V>
struct OpAddWrap : SameCarry<V, OpAddWrap<V>> {
    __device__ __forceinline__ static V identity() { return V(0); }
    __device__ __forceinline__ static V op(V a, V b) { return a + b; }
};
template <class V>
struct OpMulWrap : SameCarry<V, OpMulWrap<V>> {
    __device__ __forceinline__ static V identity() { return V(1); }
    __device__ __forceinline__ static V op(V a, V b) { return a * b; }
};
template <class V>
struct OpAndBits : SameCarry<V, OpAndBits<V>> {
    __device__ __forceinline__ static V identity() { return ~V(0); }
    __device__ __forceinline__ static V op(V a, V b) { return a & b; }
};
template <class V>
struct OpOrBits : SameCarry<V, OpOrBits<V>> {
    __device__ __forceinline__ static V identity() { return V(0); }
    __device__ __forceinline__ static V op(V a, V b) { return a | b; }
};
template <class V>
struct OpXorBits : SameCarry<V, OpXorBits<V>> {
    __device__ __forceinline__ static V identity() { return V(0); }
    __device__ __forceinline__ static V op(V a, V b) { return a ^ b; }
};
// max / min keeping the earlier of two equal values
template <class V>
struct OpMaxOf : SameCarry<V, OpMaxOf<V>> {
    __device__ __forceinline__ static V identity() { return Extremes<V>::lowest(); }
    __device__ __forceinline__ static V op(V a, V b) { return b > a ? b : a; }
};
template <class V>
struct OpMinOf : SameCarry<V, OpMinOf<V>> {
    __device__ __forceinline__ static V identity() { return Extremes<V>::highest(); }
    __device__ __forceinline__ static V op(V a, V b) { return b < a ? b : a; }
};
// Float max / min: NaN propagates (the earlier NaN wins), so -inf / +inf are
// two-sided identities; of two equal values the earlier is kept (-0.0 and
// +0.0 stay as they came).
template <class V>
struct OpMaxNaN : SameCarry<V, OpMaxNaN<V>> {
    static constexpr bool kHeavyCombine = true;
    __device__ __forceinline__ static V identity() { return Extremes<V>::lowest(); }
    __device__ __forceinline__ static V op(V a, V b) { return (a != a) ? a : (b != b) ? b : (b > a ? b : a); }
};
template <class V>
struct OpMinNaN : SameCarry<V, OpMinNaN<V>> {
    static constexpr bool kHeavyCombine = true;
    __device__ __forceinline__ static V identity() { return Extremes<V>::highest(); }
    __device__ __forceinline__ static V op(V a, V b) { return (a != a) ? a : (b != b) ? b : (b < a ? b : a); }
};
// float32: one max.NaN / min.NaN instruction (NaN in, canonical NaN out; it
// orders -0.0 below +0.0, so equal values first keep the earlier one)
__device__ __forceinline__ float fmax_nan(float a, float b) {
    float r;
    asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
    return r;
}
__device__ __forceinline__ float fmin_nan(float a, float b) {
    float r;
    asm("min.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
    return r;
}
template <>
__device__ __forceinline__ float OpMaxNaN<float>::op(float a, float b) { return a == b ? a : fmax_nan(a, b); }
template <>
__device__ __forceinline__ float OpMinNaN<float>::op(float a, float b) { return a == b ? a : fmin_nan(a, b); }

struct OpSumF64 : SameCarry<double, OpSumF64> {
    static constexpr bool kHeavyCombine = true;  // float64 adds are slow on this part
    __device__ __forceinline__ static double identity() { return 0.0; }
    __device__ __forceinline__ static double op(double a, double b) { return __dadd_rn(a, b); }
};
// (maximum, count) pairs stored as uint2 {x = int32 value bits, y = count}:
// the pair with the larger value; equal values add their counts (mod 2^32).
struct OpMaxCount : SameCarry<uint2, OpMaxCount> {
    static constexpr bool kHeavyCombine = true;
    __device__ __forceinline__ static uint2 identity() { return make_uint2(0x80000000u, 0u); }
    __device__ __forceinline__ static uint2 op(uint2 a, uint2 b) {
        const int va = (int)a.x, vb = (int)b.x;
        return vb > va ? b : (vb == va ? make_uint2(a.x, a.y + b.y) : a);
    }
};

using OpProdU32 = OpMulWrap<uint32_t>;
using OpAndU32 = OpAndBits<uint32_t>;
using OpOrU32 = OpOrBits<uint32_t>;
using OpXorU32 = OpXorBits<uint32_t>;
using OpMinI32 = OpMinOf<int32_t>;
using OpMaxU32 = OpMaxOf<uint32_t>;
using OpMinU32 = OpMinOf<uint32_t>;
using OpSumU64 = OpAddWrap<unsigned long long>;
using OpProdU64 = OpMulWrap<unsigned long long>;
using OpAndU64 = OpAndBits<unsigned long long>;
using OpOrU64 = OpOrBits<unsigned long long>;
using OpXorU64 = OpXorBits<unsigned long long>;
using OpMaxI64 = OpMaxOf<long long>;
using OpMinI64 = OpMinOf<long long>;
using OpMaxU64 = OpMaxOf<unsigned long long>;
using OpMinU64 = OpMinOf<unsigned long long>;
using OpMaxF32 = OpMaxNaN<float>;
using OpMinF32 = OpMinNaN<float>;
using OpMaxF64 = OpMaxNaN<double>;
using OpMinF64 = OpMinNaN<double>;

// Counts for the fused compaction.
struct OpCountU32 {
    using T = uint32_t;
    using C = uint32_t;
    __device__ __forceinline__ static T identity() { return 0u; }
    __device__ __forceinline__ static T op(T a, T b) { return a + b; }
    __device__ __forceinline__ static C c_identity() { return 0u; }
    __device__ __forceinline__ static C c_op(C a, C b) { return a + b; }
    __device__ __forceinline__ static C lift(T a) { return a; }
    __device__ __forceinline__ static T lower(C c) { return c; }
};

struct OpCountU64 {
    using T = uint32_t;                 // per-tile counts fit 32 bits
    using C = unsigned long long;       // running count may exceed 2^32
    __device__ __forceinline__ static T identity() { return 0u; }
    __device__ __forceinline__ static T op(T a, T b) { return a + b; }
    __device__ __forceinline__ static C c_identity() { return 0ull; }
    __device__ __forceinline__ static C c_op(C a, C b) { return a + b; }
    __device__ __forceinline__ static C lift(T a) { return a; }
    __device__ __forceinline__ static T lower(C c) { return (T)c; }
};

// ------------------------------------------------------------- bit plumbing
__device__ __forceinline__ uint32_t to_bits32(uint32_t v) { return v; }
__device__ __forceinline__ uint32_t to_bits32(int32_t v) { return (uint32_t)v; }
__device__ __forceinline__ uint32_t to_bits32(float v) { return __float_as_uint(v); }
__device__ __forceinline__ void from_bits32(uint32_t b, uint32_t& v) { v = b; }
__device__ __forceinline__ void from_bits32(uint32_t b, int32_t& v) { v = (int32_t)b; }
__device__ __forceinline__ void from_bits32(uint32_t b, float& v) { v = __uint_as_float(b); }

__device__ __forceinline__ unsigned long long to_bits64(double v) { return (unsigned long long)__double_as_longlong(v); }
__device__ __forceinline__ unsigned long long to_bits64(uint2 v) { return ((unsigned long long)v.y << 32) | v.x; }
__device__ __forceinline__ unsigned long long to_bits64(unsigned long long v) { return v; }
__device__ __forceinline__ unsigned long long to_bits64(long long v) { return (unsigned long long)v; }
__device__ __forceinline__ unsigned long long to_bits64(float2 v) {
    return ((unsigned long long)__float_as_uint(v.y) << 32) | __float_as_uint(v.x);
}
__device__ __forceinline__ void from_bits64(unsigned long long b, double& v) { v = __longlong_as_double((long long)b); }
__device__ __forceinline__ void from_bits64(unsigned long long b, uint2& v) { v = make_uint2((uint32_t)b, (uint32_t)(b >> 32)); }
__device__ __forceinline__ void from_bits64(unsigned long long b, unsigned long long& v) { v = b; }
__device__ __forceinline__ void from_bits64(unsigned long long b, long long& v) { v = (long long)b; }
__device__ __forceinline__ void from_bits64(unsigned long long b, float2& v) {
    v = make_float2(__uint_as_float((uint32_t)b), __uint_as_float((uint32_t)(b >> 32)));
}

// Warp shuffles for 4- and 8-byte value types.
template <class V>
__device__ __forceinline__ V shfl_up_v(V v, int d) {
    if constexpr (sizeof(V) == 4) {
        V r; from_bits32(__shfl_up_sync(0xffffffffu, to_bits32(v), d), r); return r;
    } else {
        unsigned long long b = to_bits64(v);
        uint32_t lo = __shfl_up_sync(0xffffffffu, (uint32_t)b, d);
        uint32_t hi = __shfl_up_sync(0xffffffffu, (uint32_t)(b >> 32), d);
        V r; from_bits64(((unsigned long long)hi << 32) | lo, r); return r;
    }
}
template <class V>
__device__ __forceinline__ V shfl_down_v(V v, int d) {
    if constexpr (sizeof(V) == 4) {
        V r; from_bits32(__shfl_down_sync(0xffffffffu, to_bits32(v), d), r); return r;
    } else {
        unsigned long long b = to_bits64(v);
        uint32_t lo = __shfl_down_sync(0xffffffffu, (uint32_t)b, d);
        uint32_t hi = __shfl_down_sync(0xffffffffu, (uint32_t)(b >> 32), d);
        V r; from_bits64(((unsigned long long)hi << 32) | lo, r); return r;
    }
}
template <class V>
__device__ __forceinline__ V shfl_idx_v(V v, int src) {
    if constexpr (sizeof(V) == 4) {
        V r; from_bits32(__shfl_sync(0xffffffffu, to_bits32(v), src), r); return r;
    } else {
        unsigned long long b = to_bits64(v);
        uint32_t lo = __shfl_sync(0xffffffffu, (uint32_t)b, src);
        uint32_t hi = __shfl_sync(0xffffffffu, (uint32_t)(b >> 32), src);
        V r; from_bits64(((unsigned long long)hi << 32) | lo, r); return r;
    }
}

__device__ __forceinline__ uint32_t lanemask_lt() { uint32_t m; asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m)); return m; }
__device__ __forceinline__ uint32_t lanemask_le() { uint32_t m; asm("mov.u32 %0, %%lanemask_le;" : "=r"(m)); return m; }

__device__ __forceinline__ unsigned long long global_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ---------------------------------------------------- look-back status words
// Strong (relaxed, gpu-scope) accesses: they bypass the non-coherent L1 so a
// spinning reader sees another SM's store.  The payload lives inside the same
// 64-bit word as its flag and epoch, so no extra ordering is needed: a word
// is read whole or not at all.
__device__ __forceinline__ unsigned long long ld_relaxed_u64(const unsigned long long* p) {
    unsigned long long v;
    asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void ld_relaxed_v2u64(const unsigned long long* p, unsigned long long& a,
                                                 unsigned long long& b) {
    asm volatile("ld.relaxed.gpu.global.v2.u64 {%0, %1}, [%2];" : "=l"(a), "=l"(b) : "l"(p) : "memory");
}
__device__ __forceinline__ void st_relaxed_u64(unsigned long long* p, unsigned long long v) {
    asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ void st_relaxed_v2u64(unsigned long long* p, unsigned long long a, unsigned long long b) {
    asm volatile("st.relaxed.gpu.global.v2.u64 [%0], {%1, %2};" ::"l"(p), "l"(a), "l"(b) : "memory");
}

// A 4-byte carry travels in one word: [payload:32 | epoch:30 | flag:2].
// An 8-byte carry travels in two words (one 16-byte store), each holding one
// half of the payload and the same [epoch | flag] tag; a reader accepts the
// pair only when both tags agree, so a half-updated pair reads as "not yet".
// A tile's status sits at word tile * stride_words (0: packed, kWords apart).
template <class C>
struct StatusIO {
    static constexpr int kWords = sizeof(C) == 4 ? 1 : 2;

    __device__ __forceinline__ static unsigned long long* slot(const LookbackCtl& lb, long long tile) {
        return lb.status + tile * (lb.stride_words ? (long long)lb.stride_words : (long long)kWords);
    }

    __device__ __forceinline__ static void publish(const LookbackCtl& lb, long long tile, unsigned flag, C v) {
        const unsigned long long tag = ((unsigned long long)lb.epoch << 2) | flag;
        if constexpr (kWords == 1) {
            st_relaxed_u64(slot(lb, tile), ((unsigned long long)to_bits32(v) << 32) | tag);
        } else {
            const unsigned long long b = to_bits64(v);
            st_relaxed_v2u64(slot(lb, tile), (b << 32) | tag, (b & 0xffffffff00000000ull) | tag);
        }
    }

    // Returns the flag (ST_INVALID when the word belongs to another call).
    __device__ __forceinline__ static unsigned read(const LookbackCtl& lb, long long tile, C& v) {
        if constexpr (kWords == 1) {
            const unsigned long long w = ld_relaxed_u64(slot(lb, tile));
            const uint32_t tag = (uint32_t)w;
            if ((tag >> 2) != lb.epoch) return ST_INVALID;
            from_bits32((uint32_t)(w >> 32), v);
            return tag & 3u;
        } else {
            unsigned long long w0, w1;
            ld_relaxed_v2u64(slot(lb, tile), w0, w1);
            const uint32_t t0 = (uint32_t)w0, t1 = (uint32_t)w1;
            if (t0 != t1 || (t0 >> 2) != lb.epoch) return ST_INVALID;
            from_bits64((w1 & 0xffffffff00000000ull) | (w0 >> 32), v);
            return t0 & 3u;
        }
    }
};

// Float-float carries (the float32 sum's (high, low) pair, and its
// segmented form, which keeps a segment flag in the low part's lowest bit)
// travel in ONE 64-bit word: the high part's 32 bits, then the low part as a
// signed 22-bit multiple of 2^-21 ulp(high) (|low| <= ulp(high)/2, so the
// multiple fits; quantisation error <= 2^-22 ulp(high) = 2^-45 |high|), a
// 7-bit epoch, the 2-bit flag and the low part's lowest bit:
//   [high:32 | lowq:22 | epoch:7 | flag:2 | lowbit:1].
// One word is read and written whole, and a one-word status measured about
// half of the float32 sum's gap to the uint32 sum on GB300 (the other half
// is the float-float arithmetic, see LowFold).  The host keeps the epoch of
// calls with this carry below 2^7 (it clears the status area when the
// workspace's epoch would pass 127).
template <>
struct StatusIO<float2> {
    static constexpr int kWords = 1;

    __device__ __forceinline__ static unsigned long long* slot(const LookbackCtl& lb, long long tile) {
        return lb.status + tile * (lb.stride_words ? (long long)lb.stride_words : 1ll);
    }
    // exponent field of the high part; the low part's scale is ulp(high) * 2^-21 = 2^(e - 171)
    __device__ __forceinline__ static int expo(float hi) { return (int)((__float_as_uint(hi) >> 23) & 0xffu); }

    __device__ __forceinline__ static void publish(const LookbackCtl& lb, long long tile, unsigned flag, float2 v) {
        const uint32_t lob = __float_as_uint(v.y);
        const int e = expo(v.x);
        int q = 0;
        if (e != 0 && e != 255) {
            // low * 2^(171 - e) by two exact power-of-two factors, each a normal
            // float (|a|, |b| <= 85; |low| <= ulp(high) / 2, so the product is at
            // most 2^20 and every step is exact), then rounded to an integer
            const int k = 171 - e, b = k >> 1, a = k - b;
            q = __float2int_rn(__fmul_rn(__fmul_rn(__uint_as_float(lob & ~1u), __uint_as_float((uint32_t)(a + 127) << 23)),
                                         __uint_as_float((uint32_t)(b + 127) << 23)));
        }
        q = max(-(1 << 21), min((1 << 21) - 1, q));
        const uint32_t lo = ((uint32_t)q << 10) | ((lb.epoch & 0x7fu) << 3) | ((flag & 3u) << 1) | (lob & 1u);
        st_relaxed_u64(slot(lb, tile), ((unsigned long long)__float_as_uint(v.x) << 32) | lo);
    }

    __device__ __forceinline__ static unsigned read(const LookbackCtl& lb, long long tile, float2& v) {
        const unsigned long long w = ld_relaxed_u64(slot(lb, tile));
        const uint32_t lo = (uint32_t)w;
        if (((lo >> 3) & 0x7fu) != lb.epoch) return ST_INVALID;
        const float hi = __uint_as_float((uint32_t)(w >> 32));
        const int q = (int)lo >> 10;  // arithmetic shift: the signed multiple
        // l = q * 2^(e - 171), rounded once, without a library call: (float)q
        // by the 1.5 * 2^23 trick (exact for |q| < 2^22), then two exact
        // power-of-two factors 2^a * 2^b = 2^(e - 171), each a normal float
        // (|a|, |b| <= 85; e = 0 and 255 carry q = 0): q * 2^a is exact, so
        // the result is rounded once, as a correctly rounded ldexpf would be.
        const int k = max(expo(hi), 1) - 171;
        const int b = k >> 1, a = k - b;
        const float qf = __fsub_rn(__int_as_float(0x4B400000 + q), 12582912.0f);
        const float l = __fmul_rn(__fmul_rn(qf, __uint_as_float((uint32_t)(a + 127) << 23)),
                                  __uint_as_float((uint32_t)(b + 127) << 23));
        v = make_float2(hi, __uint_as_float((__float_as_uint(l) & ~1u) | (lo & 1u)));
        return (lo >> 1) & 3u;
    }
};

// Record a device-side failure (first error wins).
__device__ __forceinline__ void raise_error(unsigned int* err, unsigned code) { atomicCAS(err, 0u, code); }

// Operators whose look-back may fold the aggregates after the newest
// inclusive prefix in a cheaper, lower precision L (Op::low, Op::low_op) and
// combine that sum with the prefix once (Op::with_low).  The float32 sum does:
// its aggregates are float32 chunk totals (their low parts dropped), each
// folded into exactly one prefix, so the float32 rounding of these folds adds
// at most about log2(256) * 2^-24 of the sum of |x| over the folded chunks,
// and the carried prefixes stay float-float.
template <class Op, class = void>
struct LowFold { static constexpr bool value = false; };
template <class Op>
struct LowFold<Op, std::void_t<decltype(Op::kLowFold)>> { static constexpr bool value = Op::kLowFold; };

// The low-precision accumulator type of a LowFold operator (unused otherwise).
template <class Op, bool = LowFold<Op>::value>
struct LowFoldType {
    using L = int;
    __device__ __forceinline__ static L identity() { return 0; }
};
template <class Op>
struct LowFoldType<Op, true> {
    using L = typename Op::L;
    __device__ __forceinline__ static L identity() { return Op::low_identity(); }
};

// One look-back window of a LowFold operator: the aggregates after the newest
// inclusive prefix (lane hp, entry newest_p; hp < 0: none in the window) are
// folded in the low precision into low_acc (which holds those of the newer
// windows); when the window holds the prefix, prefix (+) low_acc is left in
// acc and true returned.  Entries j >= per are unused.
template <class Op, int kMax>
__device__ __forceinline__ bool fold_window_low(const typename Op::C (&val)[kMax], int per, int newest_p, int hp,
                                                typename Op::L& low_acc, typename Op::C& acc) {
    using C = typename Op::C;
    using L = typename Op::L;
    const int lane = threadIdx.x & 31;
    L xs = Op::low_identity();
    C pv = Op::c_identity();
    if (lane >= hp) {
        const int j0 = lane == hp ? newest_p + 1 : 0;
#pragma unroll
        for (int j = 0; j < kMax; ++j) {
            if (j < per && j >= j0) xs = Op::low_op(xs, Op::low(val[j]));
            if (lane == hp && j == newest_p) pv = val[j];
        }
    }
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const L y = shfl_down_v(xs, d);
        if (lane + d < 32) xs = Op::low_op(xs, y);
    }
    low_acc = Op::low_op(shfl_idx_v(xs, 0), low_acc);
    if (hp < 0) return false;
    acc = Op::with_low(shfl_idx_v(pv, hp), low_acc);
    return true;
}

// Warp-collective decoupled look-back for tile `tile` (> 0).  A window covers
// the 32*kPer predecessors [end - 32*kPer, end): lane l reads the kPer
// consecutive tiles starting at end - 32*kPer + l*kPer, all loads issued
// back to back, so one round trip to L2 inspects 32*kPer tiles.  The window
// slides back until it holds a tile with an inclusive prefix (P).  Only the
// tiles after the newest P in the window need to be published (A or P);
// older ones are never waited for.  The newest P and every aggregate (A)
// after it are folded in tile order, older operand on the left, so
// non-commutative operators are safe.  Every wait is bounded:
// past lb.timeout_ns (or a poll cap) the warp gives up.  Returns false on
// timeout or when a predecessor is poisoned.
template <class Op, int kPer = 1>
__device__ bool lookback_prefix(const LookbackCtl& lb, long long tile, typename Op::C& prefix,
                                unsigned* windows_out = nullptr, unsigned* polls_out = nullptr) {
    using C = typename Op::C;
    constexpr int W = 32 * kPer;
    const int lane = threadIdx.x & 31;
    C acc = Op::c_identity();
    typename LowFoldType<Op>::L low_acc = LowFoldType<Op>::identity();
    long long end = tile;
    unsigned long long t_start = 0;
    unsigned polls = 0;
    unsigned sleep_ns = 16;
    while (true) {
        const long long first = end - W + (long long)lane * kPer;
        C val[kPer];
        unsigned flag[kPer];
#pragma unroll
        for (int j = 0; j < kPer; ++j) {
            val[j] = Op::c_identity();
            flag[j] = ST_PREFIX;  // tiles before 0 act as an identity prefix
            if (first + j >= 0) flag[j] = StatusIO<C>::read(lb, first + j, val[j]);
        }
        int newest_p = -1;  // index j of the newest P in this lane
#pragma unroll
        for (int j = 0; j < kPer; ++j)
            if (flag[j] == ST_PREFIX) newest_p = j;
        const uint32_t pm = __ballot_sync(0xffffffffu, newest_p >= 0);
        const int hp = pm ? 31 - __clz(pm) : -1;  // newest lane holding a P
        // only the tiles after the newest P matter: they must all be published
        bool poison = false, invalid = false;
#pragma unroll
        for (int j = 0; j < kPer; ++j) {
            const bool after = lane > hp || (lane == hp && j > newest_p);
            poison |= after && flag[j] == ST_POISON;
            invalid |= after && flag[j] == ST_INVALID;
        }
        if (__any_sync(0xffffffffu, poison)) return false;
        if (__any_sync(0xffffffffu, invalid)) {
            if (t_start == 0) t_start = global_ns();
            ++polls;
            if (polls > (1u << 26) || global_ns() - t_start > lb.timeout_ns) {
                if (lane == 0) raise_error(lb.error, DEV_LOOKBACK_TIMEOUT);
                return false;
            }
            __nanosleep(sleep_ns);
            sleep_ns = min(sleep_ns * 2u, 256u);
            continue;
        }
        if (windows_out) ++*windows_out;
        if constexpr (LowFold<Op>::value) {
            if (fold_window_low<Op, kPer>(val, kPer, newest_p, hp, low_acc, acc)) break;
        } else {
            C x = Op::c_identity();
            if (lane >= hp) {
                const int j0 = lane == hp ? newest_p : 0;
#pragma unroll
                for (int j = 0; j < kPer; ++j)
                    if (j >= j0) x = Op::c_op(x, val[j]);
            }
#pragma unroll
            for (int d = 1; d < 32; d <<= 1) {
                const C y = shfl_down_v(x, d);
                if (lane + d < 32) x = Op::c_op(x, y);
            }
            acc = Op::c_op(shfl_idx_v(x, 0), acc);
            if (pm) break;
        }
        end -= W;
    }
    if (polls_out) *polls_out = polls;
    prefix = acc;
    return true;
}

// Look-back with an adaptive window for callers that run many look-backs at
// once: the first window is 32 tiles (one status word per lane) and each
// window that holds no inclusive prefix doubles the next one, up to
// 32 * kMaxPer tiles.  Waits back off from 64 ns to 256 ns between polls.
// Same contract as lookback_prefix.  The first window covers 32 * kFirstPer
// predecessors.
template <class Op, int kMaxPer, int kFirstPer = 1>
__device__ bool lookback_prefix_adaptive(const LookbackCtl& lb, long long tile, typename Op::C& prefix,
                                         unsigned* windows_out = nullptr, unsigned* polls_out = nullptr) {
    static_assert(kFirstPer >= 1 && kFirstPer <= kMaxPer, "first window");
    using C = typename Op::C;
    const int lane = threadIdx.x & 31;
    C acc = Op::c_identity();
    typename LowFoldType<Op>::L low_acc = LowFoldType<Op>::identity();
    long long end = tile;
    int per = kFirstPer;
    unsigned long long t_start = 0;
    unsigned polls = 0;
    unsigned sleep_ns = 64;
    while (true) {
        const long long first = end - 32LL * per + (long long)lane * per;
        C val[kMaxPer];
        unsigned flag[kMaxPer];
#pragma unroll
        for (int j = 0; j < kMaxPer; ++j) {
            val[j] = Op::c_identity();
            flag[j] = ST_PREFIX;  // tiles before 0 act as an identity prefix
            if (j < per && first + j >= 0) flag[j] = StatusIO<C>::read(lb, first + j, val[j]);
        }
        int newest_p = -1;
#pragma unroll
        for (int j = 0; j < kMaxPer; ++j)
            if (j < per && flag[j] == ST_PREFIX) newest_p = j;
        const uint32_t pm = __ballot_sync(0xffffffffu, newest_p >= 0);
        const int hp = pm ? 31 - __clz(pm) : -1;
        // only the tiles after the newest P matter: they must all be published
        bool poison = false, invalid = false;
#pragma unroll
        for (int j = 0; j < kMaxPer; ++j) {
            const bool after = j < per && (lane > hp || (lane == hp && j > newest_p));
            poison |= after && flag[j] == ST_POISON;
            invalid |= after && flag[j] == ST_INVALID;
        }
        if (__any_sync(0xffffffffu, poison)) return false;
        if (__any_sync(0xffffffffu, invalid)) {
            if (t_start == 0) t_start = global_ns();
            ++polls;
            if (polls > (1u << 26) || global_ns() - t_start > lb.timeout_ns) {
                if (lane == 0) raise_error(lb.error, DEV_LOOKBACK_TIMEOUT);
                return false;
            }
            __nanosleep(sleep_ns);
            sleep_ns = min(sleep_ns * 2u, 256u);
            continue;
        }
        if (windows_out) ++*windows_out;
        if constexpr (LowFold<Op>::value) {
            if (fold_window_low<Op, kMaxPer>(val, per, newest_p, hp, low_acc, acc)) break;
        } else {
            C x = Op::c_identity();
            if (lane >= hp) {
                const int j0 = lane == hp ? newest_p : 0;
#pragma unroll
                for (int j = 0; j < kMaxPer; ++j)
                    if (j < per && j >= j0) x = Op::c_op(x, val[j]);
            }
#pragma unroll
            for (int d = 1; d < 32; d <<= 1) {
                const C y = shfl_down_v(x, d);
                if (lane + d < 32) x = Op::c_op(x, y);
            }
            acc = Op::c_op(shfl_idx_v(x, 0), acc);
            if (pm) break;
        }
        end -= 32LL * per;
        per = min(per * 2, kMaxPer);
    }
    if (polls_out) *polls_out = polls;
    prefix = acc;
    return true;
}

// --------------------------------------------------------------- tile I/O
// 16-byte vectors <-> items.
template <class T>
struct Vec {
    static constexpr int kPer = 16 / sizeof(T);
};

__device__ __forceinline__ void unpack(const uint4& r, uint32_t* v) { v[0] = r.x; v[1] = r.y; v[2] = r.z; v[3] = r.w; }
__device__ __forceinline__ void unpack(const uint4& r, int32_t* v) {
    v[0] = (int32_t)r.x; v[1] = (int32_t)r.y; v[2] = (int32_t)r.z; v[3] = (int32_t)r.w;
}
__device__ __forceinline__ void unpack(const uint4& r, float* v) {
    v[0] = __uint_as_float(r.x); v[1] = __uint_as_float(r.y); v[2] = __uint_as_float(r.z); v[3] = __uint_as_float(r.w);
}
__device__ __forceinline__ void unpack(const uint4& r, uint2* v) { v[0] = make_uint2(r.x, r.y); v[1] = make_uint2(r.z, r.w); }
__device__ __forceinline__ void unpack(const uint4& r, unsigned long long* v) {
    v[0] = ((unsigned long long)r.y << 32) | r.x; v[1] = ((unsigned long long)r.w << 32) | r.z;
}
__device__ __forceinline__ void unpack(const uint4& r, long long* v) {
    v[0] = (long long)(((unsigned long long)r.y << 32) | r.x); v[1] = (long long)(((unsigned long long)r.w << 32) | r.z);
}
__device__ __forceinline__ void unpack(const uint4& r, double* v) {
    v[0] = __hiloint2double((int)r.y, (int)r.x); v[1] = __hiloint2double((int)r.w, (int)r.z);
}

__device__ __forceinline__ uint4 pack(const uint32_t* v) { return make_uint4(v[0], v[1], v[2], v[3]); }
__device__ __forceinline__ uint4 pack(const int32_t* v) { return make_uint4((uint32_t)v[0], (uint32_t)v[1], (uint32_t)v[2], (uint32_t)v[3]); }
__device__ __forceinline__ uint4 pack(const float* v) {
    return make_uint4(__float_as_uint(v[0]), __float_as_uint(v[1]), __float_as_uint(v[2]), __float_as_uint(v[3]));
}
__device__ __forceinline__ uint4 pack(const uint2* v) { return make_uint4(v[0].x, v[0].y, v[1].x, v[1].y); }
__device__ __forceinline__ uint4 pack(const unsigned long long* v) {
    return make_uint4((uint32_t)v[0], (uint32_t)(v[0] >> 32), (uint32_t)v[1], (uint32_t)(v[1] >> 32));
}
__device__ __forceinline__ uint4 pack(const long long* v) { return pack(reinterpret_cast<const unsigned long long*>(v)); }
__device__ __forceinline__ uint4 pack(const double* v) {
    return make_uint4((uint32_t)__double2loint(v[0]), (uint32_t)__double2hiint(v[0]), (uint32_t)__double2loint(v[1]),
                      (uint32_t)__double2hiint(v[1]));
}

__device__ __forceinline__ uint4 ld_stream(const uint4* p) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p));
    return r;
}
__device__ __forceinline__ void st_stream(uint4* p, const uint4& r) {
    asm volatile("st.global.cs.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(r.x), "r"(r.y), "r"(r.z), "r"(r.w)
                 : "memory");
}

// Loader kinds.
//   LOAD_DIRECT: each thread reads its own IPT contiguous items with 16-byte loads.
//   LOAD_XPOSE : each warp reads its 32*IPT items fully coalesced (lane-contiguous
//                16-byte vectors) and transposes them to the blocked arrangement
//                through a swizzled shared-memory buffer private to the warp.
enum { LOAD_DIRECT = 0, LOAD_XPOSE = 1 };

// XOR swizzle of 16-byte chunk c inside a warp's buffer: keeps both the striped
// writes and the blocked reads (stride IPT*sizeof(T) bytes) free of bank conflicts.
__device__ __forceinline__ int swz(int c) { return c ^ ((c >> 3) & 7); }

template <class T, int IPT, int kLoad>
__device__ __forceinline__ void load_full_tile(const T* __restrict__ tile_in, T (&v)[IPT], uint4* warp_buf) {
    constexpr int NV = IPT / Vec<T>::kPer;
    const int lane = threadIdx.x & 31;
    uint4 r[NV];
    if constexpr (kLoad == LOAD_DIRECT) {
        const uint4* src = reinterpret_cast<const uint4*>(tile_in) + threadIdx.x * NV;
#pragma unroll
        for (int j = 0; j < NV; ++j) r[j] = __ldg(src + j);
    } else {
        const uint4* src = reinterpret_cast<const uint4*>(tile_in) + (threadIdx.x >> 5) * 32 * NV;
#pragma unroll
        for (int j = 0; j < NV; ++j) r[j] = ld_stream(src + j * 32 + lane);
#pragma unroll
        for (int j = 0; j < NV; ++j) warp_buf[swz(j * 32 + lane)] = r[j];
        __syncwarp();
#pragma unroll
        for (int j = 0; j < NV; ++j) r[j] = warp_buf[swz(lane * NV + j)];
    }
#pragma unroll
    for (int j = 0; j < NV; ++j) unpack(r[j], &v[j * Vec<T>::kPer]);
}

template <class T, int IPT, int kLoad>
__device__ __forceinline__ void store_full_tile(T* __restrict__ tile_out, const T (&v)[IPT], uint4* warp_buf) {
    constexpr int NV = IPT / Vec<T>::kPer;
    const int lane = threadIdx.x & 31;
    uint4 r[NV];
#pragma unroll
    for (int j = 0; j < NV; ++j) r[j] = pack(&v[j * Vec<T>::kPer]);
    if constexpr (kLoad == LOAD_DIRECT) {
        uint4* dst = reinterpret_cast<uint4*>(tile_out) + threadIdx.x * NV;
#pragma unroll
        for (int j = 0; j < NV; ++j) dst[j] = r[j];
    } else {
        __syncwarp();  // every lane has finished reading the load transpose
#pragma unroll
        for (int j = 0; j < NV; ++j) warp_buf[swz(lane * NV + j)] = r[j];
        __syncwarp();
        uint4* dst = reinterpret_cast<uint4*>(tile_out) + (threadIdx.x >> 5) * 32 * NV;
#pragma unroll
        for (int j = 0; j < NV; ++j) st_stream(dst + j * 32 + lane, warp_buf[swz(j * 32 + lane)]);
    }
}

// Partial (last) tile, or pointers that are not 16-byte aligned: element loads
// with a bound check; slots past the end hold the identity (so they do not
// change any prefix) and are never stored.
template <class T, int IPT>
__device__ __forceinline__ void load_partial_tile(const T* __restrict__ tile_in, T (&v)[IPT], long long valid, T ident) {
    const long long base = (long long)threadIdx.x * IPT;
#pragma unroll
    for (int k = 0; k < IPT; ++k) v[k] = (base + k < valid) ? tile_in[base + k] : ident;
}

template <class T, int IPT>
__device__ __forceinline__ void store_partial_tile(T* __restrict__ tile_out, const T (&v)[IPT], long long valid) {
    const long long base = (long long)threadIdx.x * IPT;
#pragma unroll
    for (int k = 0; k < IPT; ++k)
        if (base + k < valid) tile_out[base + k] = v[k];
}

}  // namespace scg
