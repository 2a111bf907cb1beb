// attn_impl.cuh -- body of the paged GQA decode attention for one work item
// (request b, KV head kvh, token chunk `split`), shared by the standalone
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
// The item runs on the first kAttnThreads threads of the CTA and synchronises
// with named barrier 1, so that the rest of a larger CTA may skip it. It
// serves the whole GQA group of Hq/Hkv query heads, so every cached K/V byte is
// read once:
//   1. the chunk's cached K and V rows (earlier tokens) are copied into shared
//      memory with cp.async (in the standalone kernel before
//      griddepcontrol.wait, so the KV read overlaps the previous kernel);
//   2. fused prologue: per-head RMSNorm of the query heads and of the new K
//      head (float32, rounded to BF16), rotate-half RoPE at position
//      ctx_len - 1 from a cos/sin table (rounded to BF16); the item whose chunk
//      holds the new token writes K/V into the cache slot and its tiles;
//   3. scores: D/8 lanes per token, 8 BF16 of K per lane, reduced over the
//      lane group with shuffles; 4. float32 max-subtracted softmax per head;
//   5. P.V with column pairs per thread, reduced over token groups;
//   6. one chunk: normalise and write BF16; several chunks: write float32
//      partials (unnormalised o, running max m, sum l) for the combine pass:
//      O = sum_s o_s e^{m_s - M} / sum_s l_s e^{m_s - M}.
#pragma once

#include "kernels.cuh"

namespace a8w8 {

constexpr int kAttnThreads = 256;
constexpr int kAttnWarps = kAttnThreads / 32;
constexpr int kGMax = 8;

// Shared memory of one item: K and V tiles (BF16), the G query rows (float),
// scores / probabilities (two-float: hi and lo planes), per-head (m, l) as
// two-float pairs. The P.V cross-group reduction reuses the K/V tiles.
__host__ __device__ inline size_t attn_item_smem_bytes(int chunk, int D) {
    return (size_t)2 * chunk * D * 2 + (size_t)kGMax * D * 4 + (size_t)2 * kGMax * chunk * 4 +
           (size_t)kGMax * 4 * 4 + 16;
}

__device__ __forceinline__ void attn_sync() {
    asm volatile("bar.sync 1, %0;" ::"n"(kAttnThreads) : "memory");
}

// Per-head RMSNorm + RoPE of one head vector held as E = D/32 elements per
// lane (elements [lane*E, lane*E + E)); the rotate-half partner of lane l is
// lane l ^ 16. Returns BF16-rounded results in y.
template <int D>
__device__ __forceinline__ void norm_rope_head(const bf16* src, const bf16* norm_w,
                                               const float* rope_row, float eps, int lane,
                                               float (&y)[D / 32]) {
    constexpr int E = D / 32;
    float x[E];
#pragma unroll
    for (int e = 0; e < E; ++e) x[e] = bf2f(ld_cg_bf16(src + lane * E + e));
    // per-head RMSNorm, correctly rounded to BF16 (see norm_bf16); the
    // float64 scalar is evaluated by lane 0 and broadcast
    f2 ss = {0.0f, 0.0f};
#pragma unroll
    for (int e = 0; e < E; ++e) f2_acc(ss, __fmul_rn(x[e], x[e]));
    ss = warp_sum_f2(ss);
    f2 inv = {0.0f, 0.0f};
    if (lane == 0) inv = rms_inv(ss, D, eps);
    inv.hi = __shfl_sync(0xffffffffu, inv.hi, 0);
    inv.lo = __shfl_sync(0xffffffffu, inv.lo, 0);
#pragma unroll
    for (int e = 0; e < E; ++e) x[e] = bf2f(norm_bf16(x[e], bf2f(norm_w[lane * E + e]), inv));
    // rotate-half RoPE, each output correctly rounded to BF16: x and its
    // partner are exact floats, cos / sin are hi + lo pairs from the table
#pragma unroll
    for (int e = 0; e < E; ++e) {
        const float partner = __shfl_xor_sync(0xffffffffu, x[e], 16);
        const int i = (lane * E + e) % (D / 2);
        const f2 c = {rope_row[i], rope_row[D + i]};
        const f2 sn = {rope_row[D / 2 + i], rope_row[3 * D / 2 + i]};
        const f2 a = f2_mulf(c, x[e]);
        const f2 b2 = f2_mulf(sn, partner);
        y[e] = bf2f(f2_to_bf16(lane < 16 ? f2_sub(a, b2) : f2_add(a, b2)));
    }
}

// One attention work item. Threads with threadIdx.x >= kAttnThreads must not
// call it. With `pdl` the cached-KV copies are issued before
// griddepcontrol.wait.
template <int D>
__device__ __forceinline__ void attn_item(const AttnParams& p, int chunk, int splits, int split,
                                          int kvh, int b, unsigned char* smem, bool pdl) {
    bf16* Ks = reinterpret_cast<bf16*>(smem);
    bf16* Vs = Ks + (size_t)chunk * D;
    float* qs = reinterpret_cast<float*>(Vs + (size_t)chunk * D);
    float* sc = qs + kGMax * D;                    // [G][chunk] hi
    float* sl = sc + (size_t)kGMax * chunk;        // [G][chunk] lo
    float* stat = sl + (size_t)kGMax * chunk;      // [G][4]: m hi, m lo, l hi, l lo
    int* s_bad_block = reinterpret_cast<int*>(stat + kGMax * 4);
    float* red = reinterpret_cast<float*>(smem);   // aliases the K/V tiles after P.V

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int G = p.Hq / p.Hkv;
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

    if (tid == 0) *s_bad_block = 0;
    attn_sync();
    constexpr int RV = D / 8;   // 16-byte vectors per row
    for (int i = tid; i < n_old * RV; i += kAttnThreads) {
        const int t = i / RV, c = i - t * RV;
        const int tok = t0 + t;
        const int blk = p.block_table[(size_t)b * p.max_blocks + tok / p.page];
        if (blk < 0 || blk >= p.num_blocks) {
            *reinterpret_cast<int4*>(Ks + (size_t)t * D + 8 * c) = make_int4(0, 0, 0, 0);
            *reinterpret_cast<int4*>(Vs + (size_t)t * D + 8 * c) = make_int4(0, 0, 0, 0);
            *s_bad_block = 1;
            continue;
        }
        const size_t off = (((size_t)blk * p.page + tok % p.page) * p.Hkv + kvh) * D + 8 * c;
        cp_async16(Ks + (size_t)t * D + 8 * c, p.k_cache + off);
        cp_async16(Vs + (size_t)t * D + 8 * c, p.v_cache + off);
    }
    cp_async_commit();

    if (pdl) {
        pdl_wait();
        pdl_trigger();
    }

    if (tid == 0) {
        if (bad_ctx) set_error(p.err, 0x4u);
        if (bad_pos) set_error(p.err, 0x10u);
    }

    // query heads (and, for the item holding the new token, its K and V)
    if (n > 0) {
        for (int task = warp; task <= G; task += kAttnWarps) {
            constexpr int E = D / 32;
            if (task < G) {
                const int h = kvh * G + task;
                const bf16* src = p.q + (size_t)b * p.q_stride + (size_t)h * D;
                float y[E];
                if (p.fused) {
                    norm_rope_head<D>(src, p.q_norm_w, p.rope + (size_t)pos * 2 * D, p.eps, lane, y);
                    if (p.tap_q_rot && split == 0) {
#pragma unroll
                        for (int e = 0; e < E; ++e)
                            p.tap_q_rot[((size_t)b * p.Hq + h) * D + lane * E + e] = f2bf(y[e]);
                    }
                } else {
#pragma unroll
                    for (int e = 0; e < E; ++e) y[e] = bf2f(ld_cg_bf16(src + lane * E + e));
                }
#pragma unroll
                for (int e = 0; e < E; ++e) qs[task * D + lane * E + e] = y[e];
            } else if (covers_new) {
                const int NQ = p.Hq * D, NK = p.Hkv * D;
                const bf16* ksrc = p.q + (size_t)b * p.q_stride + NQ + (size_t)kvh * D;
                const bf16* vsrc = p.q + (size_t)b * p.q_stride + NQ + NK + (size_t)kvh * D;
                float y[E];
                norm_rope_head<D>(ksrc, p.k_norm_w, p.rope + (size_t)pos * 2 * D, p.eps, lane, y);
                const int tr = pos - t0;
                const long slot = p.slot_mapping[b];
                const long num_slots = (long)p.num_blocks * p.page;
                const bool slot_ok = slot >= 0 && slot < num_slots;
                if (lane == 0 && slot >= num_slots) set_error(p.err, 0x1u);
#pragma unroll
                for (int e = 0; e < E; ++e) {
                    const int d = lane * E + e;
                    const bf16 kb = f2bf(y[e]);
                    const bf16 vb = ld_cg_bf16(vsrc + d);
                    Ks[(size_t)tr * D + d] = kb;
                    Vs[(size_t)tr * D + d] = vb;
                    if (slot_ok) {
                        p.k_cache[((size_t)slot * p.Hkv + kvh) * D + d] = kb;
                        p.v_cache[((size_t)slot * p.Hkv + kvh) * D + d] = vb;
                    }
                    if (p.tap_k_rot) p.tap_k_rot[((size_t)b * p.Hkv + kvh) * D + d] = kb;
                }
            }
        }
    }
    cp_async_wait_all();
    attn_sync();
    if (tid == 0 && *s_bad_block) set_error(p.err, 0x2u);

    // Scores, softmax and P.V in two-float arithmetic (see f2): q and k are
    // BF16 values, so each product q_d k_d is exact in float32 and the dot
    // product is summed as a pair; the probabilities and the weighted sum of
    // V are pairs too, so the BF16 output rounds as an evaluation in float64
    // would.
    // scores: LPT lanes per token, 8 columns each, q read from shared memory
    constexpr int LPT = D / 8;
    constexpr int TPW = 32 / LPT;
    const int j = lane % LPT, tw = lane / LPT;
    const f2 scale = {p.scale, p.scale_lo};
    if (n > 0) {
        const int step = kAttnWarps * TPW;
        const int n_pad = ((n + step - 1) / step) * step;
        for (int t = warp * TPW + tw; t < n_pad; t += step) {
            float kf[8];
            if (t < n) {
                unpack8(*reinterpret_cast<const int4*>(Ks + (size_t)t * D + 8 * j), kf);
            } else {
#pragma unroll
                for (int e = 0; e < 8; ++e) kf[e] = 0.0f;
            }
            for (int g = 0; g < G; ++g) {
                const float4 qa = *reinterpret_cast<const float4*>(qs + g * D + 8 * j);
                const float4 qb = *reinterpret_cast<const float4*>(qs + g * D + 8 * j + 4);
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
                if (j == 0 && t < n) {
                    const f2 sv = f2_mul(d, scale);
                    sc[g * chunk + t] = sv.hi;
                    sl[g * chunk + t] = sv.lo;
                }
            }
        }
    }
    attn_sync();

    // softmax over the chunk, per head: p_t = exp(s_t - m), l = sum p_t
    for (int g = warp; g < G; g += kAttnWarps) {
        f2 m = {-INFINITY, 0.0f};
        for (int t = lane; t < n; t += 32) m = f2_max(m, f2{sc[g * chunk + t], sl[g * chunk + t]});
        m = warp_max_f2(m);
        f2 l = {0.0f, 0.0f};
        for (int t = lane; t < n; t += 32) {
            const f2 e = f2_exp(f2_sub(f2{sc[g * chunk + t], sl[g * chunk + t]}, m));
            sc[g * chunk + t] = e.hi;
            sl[g * chunk + t] = e.lo;
            l = f2_add(l, e);
        }
        l = warp_sum_f2(l);
        if (lane == 0) {
            stat[4 * g] = m.hi;
            stat[4 * g + 1] = m.lo;
            stat[4 * g + 2] = l.hi;
            stat[4 * g + 3] = l.lo;
        }
    }
    attn_sync();

    // P.V: thread = (column pair, token group)
    constexpr int CP = D / 2;
    constexpr int NTG = kAttnThreads / CP;
    const int cp = tid % CP, tg = tid / CP;
    f2 o[kGMax][2];
#pragma unroll
    for (int g = 0; g < kGMax; ++g) o[g][0] = o[g][1] = f2{0.0f, 0.0f};
    for (int t = tg; t < n; t += NTG) {
        const float2 v = __bfloat1622float2(
            *reinterpret_cast<const __nv_bfloat162*>(Vs + (size_t)t * D + 2 * cp));
#pragma unroll
        for (int g = 0; g < kGMax; ++g) {
            if (g < G) {
                const f2 pr = {sc[g * chunk + t], sl[g * chunk + t]};
                o[g][0] = f2_add(o[g][0], f2_mulf(pr, v.x));
                o[g][1] = f2_add(o[g][1], f2_mulf(pr, v.y));
            }
        }
    }
    attn_sync();   // every thread is done with V: the tiles become the reduction buffer
    // red: [NTG][kGMax][2][D] (hi plane, lo plane)
#pragma unroll
    for (int g = 0; g < kGMax; ++g) {
        if (g < G) {
            float* r = red + ((size_t)tg * kGMax + g) * 2 * D;
            r[2 * cp] = o[g][0].hi;
            r[2 * cp + 1] = o[g][1].hi;
            r[D + 2 * cp] = o[g][0].lo;
            r[D + 2 * cp + 1] = o[g][1].lo;
        }
    }
    attn_sync();
    for (int i = tid; i < G * D; i += kAttnThreads) {
        const int g = i / D, d = i - g * D;
        f2 acc = {0.0f, 0.0f};
#pragma unroll
        for (int q = 0; q < NTG; ++q) {
            const float* r = red + ((size_t)q * kGMax + g) * 2 * D;
            acc = f2_add(acc, f2{r[d], r[D + d]});
        }
        const int h = kvh * G + g;
        const f2 l = {stat[4 * g + 2], stat[4 * g + 3]};
        if (splits == 1) {
            p.out[((size_t)b * p.Hq + h) * D + d] =
                n > 0 ? f2_to_bf16(f2_div(acc, l)) : __float2bfloat16_rn(0.0f);
        } else {
            // partial: o (hi, lo planes), then m and l pairs
            float* pp = p.part + (((size_t)b * p.Hq + h) * splits + split) * (2 * D + 4);
            pp[d] = n > 0 ? acc.hi : 0.0f;
            pp[D + d] = n > 0 ? acc.lo : 0.0f;
            if (d == 0) {
                pp[2 * D] = n > 0 ? stat[4 * g] : -INFINITY;
                pp[2 * D + 1] = n > 0 ? stat[4 * g + 1] : 0.0f;
                pp[2 * D + 2] = n > 0 ? l.hi : 0.0f;
                pp[2 * D + 3] = n > 0 ? l.lo : 0.0f;
            }
        }
    }
    attn_sync();   // the shared tiles may be reused by the caller afterwards
}

// Combine of split-KV partials for (request b, query head h, element d), in
// two-float arithmetic: O = sum_s o_s e^{m_s - M} / sum_s l_s e^{m_s - M}.
template <int D>
__device__ __forceinline__ void attn_combine_elem(const float* part, int splits, int Hq, int b,
                                                  int h, int d, bf16* out) {
    constexpr int S = 2 * D + 4;
    const float* pp = part + ((size_t)b * Hq + h) * splits * S;
    f2 M = {-INFINITY, 0.0f};
    for (int s = 0; s < splits; ++s)
        M = f2_max(M, f2{__ldcg(pp + (size_t)s * S + 2 * D), __ldcg(pp + (size_t)s * S + 2 * D + 1)});
    f2 L = {0.0f, 0.0f}, acc = {0.0f, 0.0f};
    if (M.hi != -INFINITY) {
        for (int s = 0; s < splits; ++s) {
            const float* q = pp + (size_t)s * S;
            const f2 m = {__ldcg(q + 2 * D), __ldcg(q + 2 * D + 1)};
            if (m.hi == -INFINITY) continue;
            const f2 w = f2_exp(f2_sub(m, M));
            L = f2_add(L, f2_mul(f2{__ldcg(q + 2 * D + 2), __ldcg(q + 2 * D + 3)}, w));
            acc = f2_add(acc, f2_mul(f2{__ldcg(q + d), __ldcg(q + D + d)}, w));
        }
    }
    out[((size_t)b * Hq + h) * D + d] =
        L.hi > 0.0f ? f2_to_bf16(f2_div(acc, L)) : __float2bfloat16_rn(0.0f);
}

}  // namespace a8w8
