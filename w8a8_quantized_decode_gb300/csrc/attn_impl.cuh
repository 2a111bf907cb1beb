// attn_impl.cuh -- body of the paged GQA decode attention for one work item
// (request b, query head h, token chunk `split`), shared by the standalone
// attention kernel and the persistent decode-step kernel.
//
// "perf(qwen3-a8w8): optimize decode scheduling and data paths" (pypto-lib PR
// #810), "BF16 KV cache": K/V are stored in BF16 with no scale tensors and
// attention loads them directly; "Add Qwen3 A8W8 L2 runner foundation"
// (pypto-serving PR #61), "Summary": block table and slot mapping address the
// pages. "[Feature] Add native Qwen3-14B A8W8 serving path" (pypto-serving
// issue #52), "Current behavior": Q and K are normalised per head and rotated
// (RoPE) before attention.
//
// The item runs on the first NT threads of the CTA and synchronises with
// named barrier 1, so that the rest of a larger CTA may skip it:
//   1. the chunk's cached K and V rows of KV head h / (Hq/Hkv) (earlier
//      tokens) are copied into shared memory with cp.async, together with the
//      norm weights and the RoPE row, before griddepcontrol.wait in the
//      standalone kernel, so these reads overlap the previous kernel;
//   2. fused prologue: per-head RMSNorm of the query head (warp 0) and of the
//      new K head (warp 1), rotate-half RoPE at position ctx_len - 1, each
//      result correctly rounded to BF16; the group's first head writes the
//      new K/V into the cache slot, every item into its own tiles;
//   3. scores: D/8 lanes per token, products of BF16 values exact in float32,
//      summed as two-float pairs and reduced over the lane group with
//      shuffles; the chunk maximum by a shared-memory atomic maximum on an
//      order-preserving 64-bit key of the pair;
//   4. softmax numerators exp(s - m), one token per thread (two-float exp);
//   5. P.V: lanes of a column pair split the tokens, two-float sums (and the
//      denominator, the sum of the numerators) combined with shuffles;
//   6. one chunk: normalise and write BF16; several chunks: write two-float
//      partials (unnormalised o, running max m, sum l) that the last chunk's
//      CTA (or a combine kernel) merges:
//      O = sum_s o_s e^{m_s - M} / sum_s l_s e^{m_s - M}.
#pragma once

#include "kernels.cuh"

namespace a8w8 {

constexpr int kAttnThreads = 256;    // the standalone / decode-layer kernel
constexpr int kTilePad = 8;          // K/V tile rows of D + 8 BF16 (16-byte aligned, fewer bank conflicts)

// Shared memory of one item (one query head): K and V tiles (BF16, padded
// rows; after P.V the region holds the in-kernel combine's scratch), the
// query row (float), scores / probabilities (two-float: hi and lo planes)
// and (m, l) as two-float pairs.
constexpr int kMaxInKernelSplits = 64;
__host__ __device__ inline size_t attn_tiles_bytes(int chunk, int D) {
    const size_t kv = (size_t)2 * chunk * (D + kTilePad) * 2;
    const size_t comb = (size_t)(2 * kMaxInKernelSplits + 2) * 4 + (size_t)(kMaxInKernelSplits + 1) * 4;
    return kv > comb ? kv : comb;
}
__host__ __device__ inline size_t attn_item_smem_bytes(int chunk, int D) {
    // ... + (m, l) pairs, then the flag (4 bytes, 4 padding) and the maximum's key (8)
    return attn_tiles_bytes(chunk, D) + (size_t)D * 4 + (size_t)2 * chunk * 4 + 4 * 4 + 16;
}

template <int NT>
__device__ __forceinline__ void attn_sync() {
    asm volatile("bar.sync 1, %0;" ::"n"(NT) : "memory");
}

template <int D>
struct HeadPre {
    static constexpr int E = D / 32;
    float qw[E], kw[E];                  // q / k norm weights
    float ch[E], sh[E], cl[E], sl[E];    // cos / sin, hi and lo parts
};

template <int D>
__device__ __forceinline__ void load_bf16_lane(const bf16* src, float (&x)[D / 32]) {
    if constexpr (D == 128) {
        const uint2 v = __ldcg(reinterpret_cast<const uint2*>(src));
        const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&v);
        const float2 a = __bfloat1622float2(h[0]), c = __bfloat1622float2(h[1]);
        x[0] = a.x;
        x[1] = a.y;
        x[2] = c.x;
        x[3] = c.y;
    } else {
        const unsigned v = __ldcg(reinterpret_cast<const unsigned*>(src));
        const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&v));
        x[0] = a.x;
        x[1] = a.y;
    }
}

template <int D>
__device__ __forceinline__ void load_head_pre(const AttnParams& p, int pos, int lane,
                                              HeadPre<D>& hp) {
    constexpr int E = D / 32;
    load_bf16_lane<D>(p.q_norm_w + lane * E, hp.qw);
    load_bf16_lane<D>(p.k_norm_w + lane * E, hp.kw);
    const float* row = p.rope + (size_t)pos * 2 * D;
    const int i0 = (lane * E) % (D / 2);
#pragma unroll
    for (int e = 0; e < E; ++e) {
        hp.ch[e] = __ldg(row + i0 + e);
        hp.sh[e] = __ldg(row + D / 2 + i0 + e);
        hp.cl[e] = __ldg(row + D + i0 + e);
        hp.sl[e] = __ldg(row + 3 * D / 2 + i0 + e);
    }
}

// Per-head RMSNorm then rotate-half RoPE of the lane's elements x, each
// output correctly rounded to BF16 (see f2): x and its partner are exact
// floats, cos / sin hi + lo pairs.
template <int D>
__device__ __forceinline__ void norm_rope_head(float (&x)[D / 32], const float (&w)[D / 32],
                                               const HeadPre<D>& hp, float eps, int lane,
                                               float (&y)[D / 32]) {
    constexpr int E = D / 32;
    f2 ss = {0.0f, 0.0f};
#pragma unroll
    for (int e = 0; e < E; ++e) f2_acc(ss, __fmul_rn(x[e], x[e]));
    const f2 inv = rms_inv(warp_sum_f2(ss), D, eps);
#pragma unroll
    for (int e = 0; e < E; ++e) x[e] = bf2f(norm_bf16(x[e], w[e], inv));
#pragma unroll
    for (int e = 0; e < E; ++e) {
        const float partner = __shfl_xor_sync(0xffffffffu, x[e], 16);
        const f2 a = f2_mulf(f2{hp.ch[e], hp.cl[e]}, x[e]);
        const f2 b2 = f2_mulf(f2{hp.sh[e], hp.sl[e]}, partner);
        y[e] = bf2f(f2_to_bf16(lane < 16 ? f2_sub(a, b2) : f2_add(a, b2)));
    }
}

// Combine of the split-KV partials of one (request b, query head h), in
// two-float arithmetic: O = sum_s o_s e^{m_s - M} / sum_s l_s e^{m_s - M}
// with M = max_s m_s. Partial layout per split: o hi plane [D], o lo plane
// [D], m (hi, lo), l (hi, lo).
// Step 1 (one warp): the split weights w_s = e^{m_s - M} into w[2s], w[2s+1]
// and L = sum_s l_s w_s into L[0], L[1].
template <int D>
__device__ __forceinline__ void combine_weights(const float* pp, int splits, float* w, float* L,
                                                int lane, int* active = nullptr,
                                                int* n_active = nullptr) {
    constexpr int S = 2 * D + 4;
    f2 M = {-INFINITY, 0.0f};
    for (int s = lane; s < splits; s += 32)
        M = f2_max(M, f2{__ldcg(pp + (size_t)s * S + 2 * D), __ldcg(pp + (size_t)s * S + 2 * D + 1)});
    M = warp_max_f2(M);
    f2 l = {0.0f, 0.0f};
    int base = 0;
    for (int s0 = 0; s0 < splits; s0 += 32) {
        const int s = s0 + lane;
        f2 ws = {0.0f, 0.0f};
        if (s < splits) {
            const float* q = pp + (size_t)s * S;
            const f2 m = {__ldcg(q + 2 * D), __ldcg(q + 2 * D + 1)};
            if (m.hi != -INFINITY) {
                ws = f2_exp(f2_sub(m, M));
                l = f2_add(l, f2_mul(f2{__ldcg(q + 2 * D + 2), __ldcg(q + 2 * D + 3)}, ws));
            }
            w[2 * s] = ws.hi;
            w[2 * s + 1] = ws.lo;
        }
        if (active) {
            // compact list of the splits with a non-zero weight
            const unsigned nz = __ballot_sync(0xffffffffu, ws.hi != 0.0f);
            if (ws.hi != 0.0f) active[base + __popc(nz & ((1u << lane) - 1u))] = s;
            base += __popc(nz);
        }
    }
    l = warp_sum_f2(l);
    if (lane == 0) {
        L[0] = l.hi;
        L[1] = l.lo;
        if (n_active) *n_active = base;
    }
}
template <int D>
__device__ __forceinline__ bf16 combine_elem(const float* pp, int splits, const float* w,
                                             const float* L, int d) {
    constexpr int S = 2 * D + 4;
    constexpr int U = 8;   // partials loaded together
    const f2 l = {L[0], L[1]};
    if (!(l.hi > 0.0f)) return __float2bfloat16_rn(0.0f);
    f2 acc = {0.0f, 0.0f};
    for (int s0 = 0; s0 < splits; s0 += U) {
        float oh[U], ol[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            oh[u] = ol[u] = 0.0f;
            if (s0 + u < splits) {
                const float* q = pp + (size_t)(s0 + u) * S;
                oh[u] = __ldcg(q + d);
                ol[u] = __ldcg(q + D + d);
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            if (s0 + u < splits) {
                const f2 ws = {w[2 * (s0 + u)], w[2 * (s0 + u) + 1]};
                if (ws.hi != 0.0f) acc = f2_add(acc, f2_mul(f2{oh[u], ol[u]}, ws));
            }
        }
    }
    return f2_to_bf16(f2_div(acc, l));
}

// Order-preserving 64-bit key of a renormalised float pair (hi, lo): the
// numeric order of the pairs is the order of the keys.
__device__ __forceinline__ unsigned ord32(float x) {
    const unsigned u = __float_as_uint(x);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float unord32(unsigned k) {
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}
__device__ __forceinline__ unsigned long long f2_key(f2 v) {
    return ((unsigned long long)ord32(v.hi) << 32) | ord32(v.lo);
}

// One attention work item, (request b, query head h, token chunk `split`),
// on the first NT threads of the CTA (the others must not call it; they are
// not synchronised with). The G query heads of a KV head are separate items
// (their K/V tiles are read once per item, from L2 after the first), so a
// batch-1 step spreads over Hq x chunks CTAs. With `pdl` the cached-KV copies
// and the other immutable operands are requested before
// griddepcontrol.wait.
template <int D, int NT>
__device__ __forceinline__ void attn_item(const AttnParams& p, int chunk, int splits, int split,
                                          int h, int b, unsigned char* smem, bool pdl) {
    constexpr int NW = NT / 32;
    constexpr int DP = D + kTilePad;
    bf16* Ks = reinterpret_cast<bf16*>(smem);
    bf16* Vs = Ks + (size_t)chunk * DP;
    float* qs = reinterpret_cast<float*>(smem + attn_tiles_bytes(chunk, D));   // [D]
    float* sc = qs + D;                            // [chunk] hi
    float* sl = sc + chunk;                        // [chunk] lo
    float* stat = sl + chunk;                      // m hi, m lo, l hi, l lo
    int* s_flag = reinterpret_cast<int*>(stat + 4);
    unsigned long long* s_mkey = reinterpret_cast<unsigned long long*>(stat + 6);

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int G = p.Hq / p.Hkv;
    const int kvh = h / G;
    const bool lead = h - kvh * G == 0;            // the head that writes the new K/V
    const int t0 = split * chunk;
    const int max_ctx = p.max_blocks * p.page;
    const int ctx_raw = p.ctx_lens[b];
    const bool bad_ctx = ctx_raw < 0 || ctx_raw > max_ctx;
    const int pos = ctx_raw - 1;
    const bool bad_pos = p.fused && !bad_ctx && ctx_raw > 0 && pos >= p.max_pos;
    const int ctx = (bad_ctx || bad_pos) ? 0 : ctx_raw;
    const int t1 = min(t0 + chunk, ctx);
    const int n = max(t1 - t0, 0);
    const bool covers_new = p.fused && ctx > 0 && pos >= t0 && pos < t0 + chunk;
    const int n_old = covers_new ? n - 1 : n;
    // In-kernel combine: only the chunks that hold tokens take part; a lone
    // chunk writes the output itself.
    const int active = p.tickets ? max(1, (ctx + chunk - 1) / chunk) : splits;
    if (split >= active) return;   // the whole CTA, before any barrier
    const bool single = active == 1;

    if (tid == 0) {
        *s_flag = 0;
        *s_mkey = 0ull;   // below every score's key
    }
    attn_sync<NT>();
    constexpr int RV = D / 8;   // 16-byte vectors per row
    for (int i = tid; i < n_old * RV; i += NT) {
        const int t = i / RV, c = i - t * RV;
        const int tok = t0 + t;
        const int blk = p.block_table[(size_t)b * p.max_blocks + tok / p.page];
        if (blk < 0 || blk >= p.num_blocks) {
            *reinterpret_cast<int4*>(Ks + (size_t)t * DP + 8 * c) = make_int4(0, 0, 0, 0);
            *reinterpret_cast<int4*>(Vs + (size_t)t * DP + 8 * c) = make_int4(0, 0, 0, 0);
            *s_flag = 1;
            continue;
        }
        const size_t off = (((size_t)blk * p.page + tok % p.page) * p.Hkv + kvh) * D + 8 * c;
        cp_async16(Ks + (size_t)t * DP + 8 * c, p.k_cache + off);
        cp_async16(Vs + (size_t)t * DP + 8 * c, p.v_cache + off);
    }
    cp_async_commit();
    HeadPre<D> hp;
    if (p.fused && n > 0 && warp < 2) load_head_pre<D>(p, pos < p.max_pos ? pos : 0, lane, hp);

    if (pdl) {
        pdl_wait();
        pdl_trigger();
    }

    if (tid == 0) {
        if (bad_ctx) set_error(p.err, 0x4u);
        if (bad_pos) set_error(p.err, 0x10u);
    }

    // warp 0: the query head; warp 1: the new token's K (norm + RoPE) and V
    constexpr int E = D / 32;
    if (n > 0 && warp == 0) {
        const bf16* src = p.q + (size_t)b * p.q_stride + (size_t)h * D;
        float x[E], y[E];
        load_bf16_lane<D>(src + lane * E, x);
        if (p.fused) {
            norm_rope_head<D>(x, hp.qw, hp, p.eps, lane, y);
            if (p.tap_q_rot && split == 0) {
#pragma unroll
                for (int e = 0; e < E; ++e)
                    p.tap_q_rot[((size_t)b * p.Hq + h) * D + lane * E + e] = f2bf(y[e]);
            }
        } else {
#pragma unroll
            for (int e = 0; e < E; ++e) y[e] = x[e];
        }
#pragma unroll
        for (int e = 0; e < E; ++e) qs[lane * E + e] = y[e];
    } else if (n > 0 && warp == 1 && covers_new) {
        const int NQ = p.Hq * D, NK = p.Hkv * D;
        const bf16* ksrc = p.q + (size_t)b * p.q_stride + NQ + (size_t)kvh * D;
        const bf16* vsrc = p.q + (size_t)b * p.q_stride + NQ + NK + (size_t)kvh * D;
        float x[E], vv[E], y[E];
        load_bf16_lane<D>(ksrc + lane * E, x);
        load_bf16_lane<D>(vsrc + lane * E, vv);
        norm_rope_head<D>(x, hp.kw, hp, p.eps, lane, y);
        const int tr = pos - t0;
        const long slot = p.slot_mapping[b];
        const long num_slots = (long)p.num_blocks * p.page;
        const bool slot_ok = lead && slot >= 0 && slot < num_slots;
        if (lead && lane == 0 && slot >= num_slots) set_error(p.err, 0x1u);
#pragma unroll
        for (int e = 0; e < E; ++e) {
            const int d = lane * E + e;
            const bf16 kb = f2bf(y[e]);
            const bf16 vb = f2bf(vv[e]);
            Ks[(size_t)tr * DP + d] = kb;
            Vs[(size_t)tr * DP + d] = vb;
            if (slot_ok) {
                p.k_cache[((size_t)slot * p.Hkv + kvh) * D + d] = kb;
                p.v_cache[((size_t)slot * p.Hkv + kvh) * D + d] = vb;
            }
            if (lead && p.tap_k_rot) p.tap_k_rot[((size_t)b * p.Hkv + kvh) * D + d] = kb;
        }
    }
    cp_async_wait_all();
    attn_sync<NT>();
    if (tid == 0 && *s_flag) set_error(p.err, 0x2u);

    // Scores, softmax and P.V in two-float arithmetic (see f2): q and k are
    // BF16 values, so each product q_d k_d is exact in float32 and the dot
    // product is summed as a pair; the probabilities and the weighted sum of
    // V are pairs too, so the BF16 output rounds as an evaluation in float64
    // would.
    // scores: one token per LPT lanes, 8 columns per lane
    constexpr int LPT = D / 8;
    constexpr int PPW = 32 / LPT;
    const f2 scale = {p.scale, p.scale_lo};
    {
        const int j = lane % LPT, pw = lane / LPT;
        const float4 qa = *reinterpret_cast<const float4*>(qs + 8 * j);
        const float4 qb = *reinterpret_cast<const float4*>(qs + 8 * j + 4);
        const int step = NW * PPW;
        const int n_pad = (n + step - 1) / step * step;
        for (int t = warp * PPW + pw; t < n_pad; t += step) {
            const bool ok = t < n;
            float kf[8];
            unpack8(*reinterpret_cast<const int4*>(Ks + (size_t)(ok ? t : 0) * DP + 8 * j), kf);
            f2 d = f2_make(__fmul_rn(qa.x, kf[0]));
            f2_acc(d, __fmul_rn(qa.y, kf[1]));
            f2_acc(d, __fmul_rn(qa.z, kf[2]));
            f2_acc(d, __fmul_rn(qa.w, kf[3]));
            f2_acc(d, __fmul_rn(qb.x, kf[4]));
            f2_acc(d, __fmul_rn(qb.y, kf[5]));
            f2_acc(d, __fmul_rn(qb.z, kf[6]));
            f2_acc(d, __fmul_rn(qb.w, kf[7]));
#pragma unroll
            for (int o = LPT / 2; o > 0; o >>= 1) {
                f2 r;
                r.hi = __shfl_xor_sync(0xffffffffu, d.hi, o);
                r.lo = __shfl_xor_sync(0xffffffffu, d.lo, o);
                d = f2_add(d, r);
            }
            if (j == 0 && ok) {
                const f2 sv = f2_mul(d, scale);
                sc[t] = sv.hi;
                sl[t] = sv.lo;
                atomicMax(s_mkey, f2_key(sv));   // the chunk maximum m
            }
        }
    }
    attn_sync<NT>();

    // softmax numerators p_t = exp(s_t - m), one token per thread; their sum
    // l is formed in the P.V reduction below
    {
        const unsigned long long mk = *s_mkey;
        const f2 m = {unord32((unsigned)(mk >> 32)), unord32((unsigned)mk)};
        if (tid == 0) {
            stat[0] = m.hi;
            stat[1] = m.lo;
        }
        for (int t = tid; t < n; t += NT) {
            const f2 e = f2_exp(f2_sub(f2{sc[t], sl[t]}, m));
            sc[t] = e.hi;
            sl[t] = e.lo;
        }
    }
    attn_sync<NT>();

    // P.V: TG consecutive lanes share a column pair and split the tokens;
    // their sums are combined with shuffles
    {
        constexpr int CP = D / 2;
        constexpr int TG = NT / CP;
        static_assert(TG >= 1 && TG <= 32 && (TG & (TG - 1)) == 0, "token groups");
        const int cp = tid / TG, tg = tid % TG;
        f2 o0 = {0.0f, 0.0f}, o1 = {0.0f, 0.0f}, l = {0.0f, 0.0f};
        for (int t = tg; t < n; t += TG) {
            const float2 v = __bfloat1622float2(
                *reinterpret_cast<const __nv_bfloat162*>(Vs + (size_t)t * DP + 2 * cp));
            const f2 pr = {sc[t], sl[t]};
            o0 = f2_add(o0, f2_mulf(pr, v.x));
            o1 = f2_add(o1, f2_mulf(pr, v.y));
            l = f2_add(l, pr);
        }
#pragma unroll
        for (int o = TG / 2; o > 0; o >>= 1) {
            f2 r;
            r.hi = __shfl_xor_sync(0xffffffffu, o0.hi, o);
            r.lo = __shfl_xor_sync(0xffffffffu, o0.lo, o);
            o0 = f2_add(o0, r);
            r.hi = __shfl_xor_sync(0xffffffffu, o1.hi, o);
            r.lo = __shfl_xor_sync(0xffffffffu, o1.lo, o);
            o1 = f2_add(o1, r);
            r.hi = __shfl_xor_sync(0xffffffffu, l.hi, o);
            r.lo = __shfl_xor_sync(0xffffffffu, l.lo, o);
            l = f2_add(l, r);
        }
        if (tg == 0) {
            if (single) {
                bf16* out = p.out + ((size_t)b * p.Hq + h) * D + 2 * cp;
                out[0] = n > 0 ? f2_to_bf16(f2_div(o0, l)) : __float2bfloat16_rn(0.0f);
                out[1] = n > 0 ? f2_to_bf16(f2_div(o1, l)) : __float2bfloat16_rn(0.0f);
            } else {
                // partial: o (hi, lo planes), then m and l pairs
                float* pp = p.part + (((size_t)b * p.Hq + h) * splits + split) * (2 * D + 4);
                pp[2 * cp] = n > 0 ? o0.hi : 0.0f;
                pp[2 * cp + 1] = n > 0 ? o1.hi : 0.0f;
                pp[D + 2 * cp] = n > 0 ? o0.lo : 0.0f;
                pp[D + 2 * cp + 1] = n > 0 ? o1.lo : 0.0f;
                if (cp == 0) {
                    pp[2 * D] = n > 0 ? stat[0] : -INFINITY;
                    pp[2 * D + 1] = n > 0 ? stat[1] : 0.0f;
                    pp[2 * D + 2] = n > 0 ? l.hi : 0.0f;
                    pp[2 * D + 3] = n > 0 ? l.lo : 0.0f;
                }
            }
        }
    }
    if (!single && p.tickets) {
        // the last CTA of this (request, query head) to finish combines the
        // partials (no CTA waits for another)
        __threadfence();
        attn_sync<NT>();
        if (tid == 0) {
            unsigned* tk = p.tickets + (size_t)b * p.Hq + h;
            const unsigned prev = atomicAdd(tk, 1u);
            *s_flag = prev == (unsigned)(active - 1);
            if (*s_flag) *tk = 0u;   // ready for the next launch
        }
        attn_sync<NT>();
        if (*s_flag) {
            __threadfence();
            // split weights and the active splits (warp 0), in the tile region
            float* cw = reinterpret_cast<float*>(smem);            // [splits][2]
            float* cl = cw + 2 * kMaxInKernelSplits;               // [2]
            int* act = reinterpret_cast<int*>(cl + 2);             // [splits]
            int* nact = act + kMaxInKernelSplits;                  // [1]
            const float* pb = p.part + ((size_t)b * p.Hq + h) * splits * (2 * D + 4);
            if (warp == 0) combine_weights<D>(pb, active, cw, cl, lane, act, nact);
            attn_sync<NT>();
            constexpr int KA = 4;   // active splits per round of loads
            for (int d = tid; d < D; d += NT) {
                f2 acc = {0.0f, 0.0f};
                for (int k0 = 0; k0 < *nact; k0 += KA) {
                    float oh[KA], ol[KA];
#pragma unroll
                    for (int k = 0; k < KA; ++k) {
                        oh[k] = ol[k] = 0.0f;
                        if (k0 + k < *nact) {
                            const float* q = pb + (size_t)act[k0 + k] * (2 * D + 4);
                            oh[k] = __ldcg(q + d);
                            ol[k] = __ldcg(q + D + d);
                        }
                    }
#pragma unroll
                    for (int k = 0; k < KA; ++k) {
                        if (k0 + k < *nact) {
                            const int sp = act[k0 + k];
                            acc = f2_add(acc, f2_mul(f2{oh[k], ol[k]}, f2{cw[2 * sp], cw[2 * sp + 1]}));
                        }
                    }
                }
                const f2 l = {cl[0], cl[1]};
                p.out[((size_t)b * p.Hq + h) * D + d] =
                    l.hi > 0.0f ? f2_to_bf16(f2_div(acc, l)) : __float2bfloat16_rn(0.0f);
            }
        }
    }
    attn_sync<NT>();   // the shared tiles may be reused by the caller afterwards
}

}  // namespace a8w8
