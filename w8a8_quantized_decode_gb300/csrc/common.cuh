// common.cuh -- device helpers shared by the A8W8 decode kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace a8w8 {

typedef __nv_bfloat16 bf16;

// ---------------------------------------------------------------------------
// Programmatic dependent launch. A kernel launched with programmatic stream
// serialization may start while its predecessor is still running; it must
// call pdl_wait() before it reads anything the predecessor writes and before
// it writes anything. Every kernel here reads only immutable inputs (weights,
// cached K/V of earlier tokens, tables) before that point. In a kernel
// launched without the attribute both instructions are no-ops.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// 16-byte streaming load of data read once (weights): bypasses L1.
__device__ __forceinline__ int4 ld_stream_v4(const void* p) {
    int4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.s32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

// 16-byte load through the read-only path, for data that no kernel writes
// (weights, tables).
__device__ __forceinline__ int4 ld_nc_v4(const void* p) {
    return __ldg(reinterpret_cast<const int4*>(p));
}

// 16-byte load from L2, bypassing L1, for data produced on the device
// (activations, partials): inside one long-running kernel an SM's L1 may
// still hold a line that another SM has since rewritten.
__device__ __forceinline__ int4 ld_cg_v4(const void* p) {
    return __ldcg(reinterpret_cast<const int4*>(p));
}
__device__ __forceinline__ bf16 ld_cg_bf16(const bf16* p) {
    unsigned short u = __ldcg(reinterpret_cast<const unsigned short*>(p));
    return __ushort_as_bfloat16(u);
}

// Asynchronous 16-byte global -> shared copy (cp.async, L2 only).
__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
    unsigned s = static_cast<unsigned>(__cvta_generic_to_shared(smem));
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(s), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }
// Same copy with a 32-bit shared-space destination address and an L2 cache
// policy (weights streamed once: evict-first, so that the small operands
// read by every step stay resident in L2).
__device__ __forceinline__ void cp_async16_s(uint32_t s, const void* gmem, uint64_t policy) {
    asm volatile("cp.async.cg.shared.global.L2::cache_hint [%0], [%1], 16, %2;" ::"r"(s), "l"(gmem),
                 "l"(policy)
                 : "memory");
}
// Wait until at most N of this thread's most recent copy groups are pending.
template <int N>
__device__ __forceinline__ void cp_async_wait_group() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ int4 lds_v4(uint32_t s) {
    int4 r;
    asm volatile("ld.shared.v4.s32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "r"(s));
    return r;
}

// L2 policy for data read once per step (weights): evict first.
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}
__device__ __forceinline__ int warp_sum_i(int v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

__device__ __forceinline__ float bf2f(bf16 v) { return __bfloat162float(v); }
__device__ __forceinline__ bf16 f2bf(float v) { return __float2bfloat16_rn(v); }

// Unpack 8 BF16 values held in an int4.
__device__ __forceinline__ void unpack8(const int4& v, float (&f)[8]) {
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        float2 t = __bfloat1622float2(h[i]);
        f[2 * i] = t.x;
        f[2 * i + 1] = t.y;
    }
}

// Per-row INT8 code of x with row scale s: clamp(rne(x / s), -127, 127) with
// x / s the IEEE float32 quotient; s == 0 gives 0. The quotient is formed
// without a division instruction, from R = RN(1 / s) (quant_recip, once per
// row): q0 = RN(x R), then one correction by the exact remainder x - q0 s
// (an FMA), q = RN(q0 + (x - q0 s) R), which equals RN(x / s) (Markstein's
// theorem, e.g. Muller et al., Handbook of Floating-Point Arithmetic, 2nd
// ed., section 4.7). Where R overflows (s below 2^-126) the division is
// used as is.
__device__ __forceinline__ float quant_recip(float s) { return s == 0.0f ? 0.0f : __frcp_rn(s); }
__device__ __forceinline__ int quant_code(float x, float s, float R) {
    if (s == 0.0f) return 0;
    float q;
    if (isfinite(R)) {
        const float q0 = __fmul_rn(x, R);
        q = __fmaf_rn(__fmaf_rn(-q0, s, x), R, q0);
    } else {
        q = __fdiv_rn(x, s);
    }
    return max(-127, min(127, __float2int_rn(q)));
}

// ---------------------------------------------------------------------------
// Two-float ("double-float") arithmetic. Every floating-point stage whose
// result is rounded to BF16 (the norms, RoPE, SiLU, attention) is evaluated
// as an unevaluated pair hi + lo carrying about 44-48 significant bits, so
// that its BF16 rounding agrees with an evaluation in float64 (and with the
// exact real value) except when that value lies within ~2^-40 (relative) of
// a rounding boundary. Building blocks (Dekker 1971; Knuth, TAOCP vol. 2):
// TwoSum and FastTwoSum give the exact rounding error of a sum, an FMA the
// exact rounding error of a product.
// ---------------------------------------------------------------------------
struct f2 {
    float hi, lo;
};

__device__ __forceinline__ f2 f2_make(float a) { return f2{a, 0.0f}; }
// Knuth's TwoSum: s + e == a + b exactly, s = fl(a + b).
__device__ __forceinline__ void two_sum(float a, float b, float& s, float& e) {
    s = __fadd_rn(a, b);
    const float bb = __fsub_rn(s, a);
    e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
}
// Dekker's FastTwoSum (|a| >= |b| or a == 0): the renormalised pair. A zero
// b leaves a untouched, so that a signed zero keeps its sign.
__device__ __forceinline__ f2 fast_two_sum(float a, float b) {
    f2 r;
    r.hi = b == 0.0f ? a : __fadd_rn(a, b);
    r.lo = __fsub_rn(b, __fsub_rn(r.hi, a));
    return r;
}
// a += v (v a float), without renormalisation (a few terms at a time).
__device__ __forceinline__ void f2_acc(f2& a, float v) {
    float s, e;
    two_sum(a.hi, v, s, e);
    a.hi = s;
    a.lo = __fadd_rn(a.lo, e);
}
__device__ __forceinline__ f2 f2_add(f2 a, f2 b) {
    float s, e;
    two_sum(a.hi, b.hi, s, e);
    e = __fadd_rn(e, __fadd_rn(a.lo, b.lo));
    return fast_two_sum(s, e);
}
__device__ __forceinline__ f2 f2_addf(f2 a, float b) {
    float s, e;
    two_sum(a.hi, b, s, e);
    return fast_two_sum(s, __fadd_rn(e, a.lo));
}
__device__ __forceinline__ f2 f2_neg(f2 a) { return f2{-a.hi, -a.lo}; }
__device__ __forceinline__ f2 f2_sub(f2 a, f2 b) { return f2_add(a, f2_neg(b)); }
// Exact product of two floats as a pair.
__device__ __forceinline__ f2 two_prod(float a, float b) {
    f2 r;
    r.hi = __fmul_rn(a, b);
    r.lo = __fmaf_rn(a, b, -r.hi);
    return r;
}
__device__ __forceinline__ f2 f2_mulf(f2 a, float b) {
    f2 p = two_prod(a.hi, b);
    return fast_two_sum(p.hi, __fmaf_rn(a.lo, b, p.lo));
}
__device__ __forceinline__ f2 f2_mul(f2 a, f2 b) {
    f2 p = two_prod(a.hi, b.hi);
    float e = __fmaf_rn(a.hi, b.lo, p.lo);
    e = __fmaf_rn(a.lo, b.hi, e);
    return fast_two_sum(p.hi, e);
}
// a / b: one correction of the float quotient by the exact remainder.
__device__ __forceinline__ f2 f2_div(f2 a, f2 b) {
    const float q1 = __fdiv_rn(a.hi, b.hi);
    const f2 r = f2_sub(a, f2_mulf(b, q1));
    const float q2 = __fdiv_rn(r.hi, b.hi);
    return fast_two_sum(q1, q2);
}
// Ordering of pairs (both renormalised).
__device__ __forceinline__ bool f2_gt(f2 a, f2 b) { return a.hi > b.hi || (a.hi == b.hi && a.lo > b.lo); }
__device__ __forceinline__ f2 f2_max(f2 a, f2 b) { return f2_gt(b, a) ? b : a; }
__device__ __forceinline__ f2 warp_sum_f2(f2 v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        f2 t;
        t.hi = __shfl_xor_sync(0xffffffffu, v.hi, o);
        t.lo = __shfl_xor_sync(0xffffffffu, v.lo, o);
        v = f2_add(v, t);
    }
    return v;
}
__device__ __forceinline__ f2 warp_max_f2(f2 v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        f2 t;
        t.hi = __shfl_xor_sync(0xffffffffu, v.hi, o);
        t.lo = __shfl_xor_sync(0xffffffffu, v.lo, o);
        v = f2_max(v, t);
    }
    return v;
}
// 1 / sqrt(s), s > 0: the float estimate refined by one Newton step
// y' = y + y (1 - s y^2) / 2 with the residual formed exactly.
__device__ __forceinline__ f2 f2_rsqrt(f2 s) {
    const float y = rsqrtf(s.hi);
    const f2 t = f2_mul(s, two_prod(y, y));
    const float e = __fsub_rn(__fsub_rn(1.0f, t.hi), t.lo);   // 1 - t.hi is exact
    return fast_two_sum(y, __fmul_rn(__fmul_rn(y, e), 0.5f));
}
// exp(x) for x.hi <= 88 (underflows to 0 below about -103): x = k ln2 + r,
// exp(r) = (1 + p)^(2^8) with p = expm1(r / 2^8) from its Taylor series to
// the fourth power, squared eight times in expm1 form (1 + p)^2 = 1 + (2p +
// p^2); then scaled by 2^k.
static __device__ __noinline__ f2 f2_exp(f2 x) {
    if (x.hi < -104.0f) return f2{0.0f, 0.0f};
    if (x.hi > 88.5f) return f2{INFINITY, 0.0f};
    const float k = rintf(__fmul_rn(x.hi, 1.44269504088896341f));
    const f2 ln2 = {0.693147182464599609375f, -1.904654323148236e-09f};   // ln 2 = hi + lo
    const f2 r = f2_sub(x, f2_mulf(ln2, k));
    const f2 t = f2{__fmul_rn(r.hi, 0.00390625f), __fmul_rn(r.lo, 0.00390625f)};   // r / 2^8
    const f2 t2 = f2_mul(t, t);
    const float t3 = __fmul_rn(t2.hi, t.hi);
    const float tail = __fmaf_rn(__fmul_rn(t3, t.hi), 1.0f / 24.0f, __fmul_rn(t3, 1.0f / 6.0f));
    f2 p = f2_addf(f2_add(t, f2{__fmul_rn(t2.hi, 0.5f), __fmul_rn(t2.lo, 0.5f)}), tail);
#pragma unroll 1
    for (int i = 0; i < 8; ++i) p = f2_add(f2{__fmul_rn(p.hi, 2.0f), __fmul_rn(p.lo, 2.0f)}, f2_mul(p, p));
    const f2 e = f2_addf(p, 1.0f);
    const int ki = (int)k;
    return f2{ldexpf(e.hi, ki), ldexpf(e.lo, ki)};
}
// BF16 nearest-even rounding of the value hi + lo.
__device__ __forceinline__ bf16 f2_to_bf16(f2 v) {
    const f2 n = fast_two_sum(v.hi, v.lo);       // |n.lo| <= ulp(n.hi) / 2
    const unsigned u = __float_as_uint(n.hi);
    if ((u & 0xFFFFu) == 0x8000u && n.lo != 0.0f && isfinite(n.hi)) {
        // n.hi is a midpoint between two BF16 values: n.lo decides
        const bool away = (n.lo > 0.0f) == (n.hi > 0.0f);
        return __ushort_as_bfloat16((unsigned short)((u >> 16) + (away ? 1u : 0u)));
    }
    return __float2bfloat16_rn(n.hi);
}

// RMSNorm pieces. Every x*x of a BF16 x is exact in float32, so a row's sum
// of squares is accumulated exactly enough with f2_acc; the scale
// 1 / sqrt(ss / n + eps) is formed in two-float arithmetic; and x * w (two
// 8-bit significands) is exact in float32, so the normalised value
// x * w * scale needs one two-float product.
__device__ __forceinline__ f2 rms_inv(f2 ss, int n, float eps) {
    return f2_rsqrt(f2_addf(f2_div(ss, f2_make((float)n)), eps));
}
__device__ __forceinline__ bf16 norm_bf16(float x, float w, f2 inv) {
    return f2_to_bf16(f2_mulf(inv, __fmul_rn(x, w)));
}
// The same rounding of xw * inv for an exact float32 xw (= x w), taking the
// float product p = RN(xw inv.hi) where it decides: the exact value differs
// from p by at most 1.5 float32 units (the product's rounding error and
// xw inv.lo), and BF16 rounding changes only at the midpoints between BF16
// values, where the low 16 bits of a float are 0x8000. Away from them
// (more than 4 units) and for normal finite p, RN_bf16(p) is the answer;
// otherwise the two-float product decides.
__device__ __forceinline__ bf16 norm_bf16_fast(float xw, f2 inv) {
    const float pr = __fmul_rn(xw, inv.hi);
    const unsigned u = __float_as_uint(pr);
    const unsigned ex = u & 0x7F800000u;
    const unsigned d = (u & 0xFFFFu) - 0x7FFCu;   // < 9 within 4 units of the midpoint
    if (d >= 9u && ex != 0u && ex != 0x7F800000u) return __float2bfloat16_rn(pr);
    return f2_to_bf16(f2_mulf(inv, xw));
}

// act = RN_bf16(silu(g) u) for float32 g, u: g u / (1 + e) for g >= 0 and
// g u e / (1 + e) for g < 0, e = exp(-|g|), evaluated in two-float
// arithmetic (f2_exp, f2_div) so that the BF16 rounding is that of the exact
// value. A float32 evaluation decides first where it can: with expf within a
// few units of its result, the three float roundings and e <= 1, it is within
// about 10 float32 units of the exact value, so where it lies more than 64
// units from a BF16 midpoint (low 16 bits 0x8000), is normal and finite, its
// own BF16 rounding is the exact value's; elsewhere (about 0.2 % of values)
// the two-float form decides.
__device__ __forceinline__ bf16 swiglu_bf16(float g, float u) {
    {
        const float ef = expf(-fabsf(g));
        float r = __fdiv_rn(__fmul_rn(g, u), __fadd_rn(1.0f, ef));
        if (g < 0.0f) r = __fmul_rn(r, ef);
        const unsigned ur = __float_as_uint(r);
        const unsigned ex = ur & 0x7F800000u;
        const unsigned d = (ur & 0xFFFFu) - (0x8000u - 64u);   // < 129 near the midpoint
        // (g > -80: for g < 0 the result is scaled by e, which must be a
        // normal float, not a subnormal with few significant bits)
        if (d >= 129u && ex != 0u && ex != 0x7F800000u && g > -80.0f) return __float2bfloat16_rn(r);
    }
    const f2 e = f2_exp(f2_make(-fabsf(g)));
    f2 num = two_prod(g, u);
    if (g < 0.0f) num = f2_mul(num, e);
    return f2_to_bf16(f2_div(num, f2_addf(e, 1.0f)));
}

__device__ __forceinline__ void set_error(unsigned* err, unsigned bit) {
    if (err) atomicOr(err, bit);
}

}  // namespace a8w8
