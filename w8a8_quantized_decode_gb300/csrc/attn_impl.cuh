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

__host__ __device__ inline size_t attn_item_smem_bytes(int chunk, int D) {
    return (size_t)2 * chunk * D * 2 + (size_t)kGMax * D * 4 + (size_t)kGMax * chunk * 4 +
           (size_t)kGMax * 2 * 4 + 16;
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
    float ss = 0.0f;
#pragma unroll
    for (int e = 0; e < E; ++e) ss += x[e] * x[e];
    ss = warp_sum(ss);
    const float inv = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(__fdiv_rn(ss, (float)D), eps)));
#pragma unroll
    for (int e = 0; e < E; ++e)
        x[e] = bf2f(f2bf(__fmul_rn(__fmul_rn(x[e], inv), bf2f(norm_w[lane * E + e]))));
#pragma unroll
    for (int e = 0; e < E; ++e) {
        const float partner = __shfl_xor_sync(0xffffffffu, x[e], 16);
        const int i = (lane * E + e) % (D / 2);
        const float c = rope_row[i], s = rope_row[D / 2 + i];
        float r;
        if (lane < 16) r = __fsub_rn(__fmul_rn(x[e], c), __fmul_rn(partner, s));
        else r = __fadd_rn(__fmul_rn(x[e], c), __fmul_rn(partner, s));
        y[e] = bf2f(f2bf(r));
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
    float* sc = qs + kGMax * D;
    float* stat = sc + (size_t)kGMax * chunk;
    int* s_bad_block = reinterpret_cast<int*>(stat + kGMax * 2);
    float* red = reinterpret_cast<float*>(smem);   // aliases Ks once the scores are done

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
                    norm_rope_head<D>(src, p.q_norm_w, p.rope + (size_t)pos * D, p.eps, lane, y);
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
                norm_rope_head<D>(ksrc, p.k_norm_w, p.rope + (size_t)pos * D, p.eps, lane, y);
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

    // scores: q read from shared memory (keeps the item within 64 registers)
    constexpr int LPT = D / 8;
    constexpr int TPW = 32 / LPT;
    const int j = lane % LPT, tw = lane / LPT;
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
                float d = 0.0f;
                d = fmaf(qa.x, kf[0], d);
                d = fmaf(qa.y, kf[1], d);
                d = fmaf(qa.z, kf[2], d);
                d = fmaf(qa.w, kf[3], d);
                d = fmaf(qb.x, kf[4], d);
                d = fmaf(qb.y, kf[5], d);
                d = fmaf(qb.z, kf[6], d);
                d = fmaf(qb.w, kf[7], d);
#pragma unroll
                for (int o = LPT / 2; o > 0; o >>= 1) d += __shfl_xor_sync(0xffffffffu, d, o);
                if (j == 0 && t < n) sc[g * chunk + t] = d * p.scale;
            }
        }
    }
    attn_sync();

    // softmax over the chunk, per head
    for (int g = warp; g < G; g += kAttnWarps) {
        float m = -INFINITY;
        for (int t = lane; t < n; t += 32) m = fmaxf(m, sc[g * chunk + t]);
        m = warp_max(m);
        float l = 0.0f;
        for (int t = lane; t < n; t += 32) {
            const float e = expf(sc[g * chunk + t] - m);
            sc[g * chunk + t] = e;
            l += e;
        }
        l = warp_sum(l);
        if (lane == 0) {
            stat[2 * g] = m;
            stat[2 * g + 1] = l;
        }
    }
    attn_sync();

    // P.V: thread = (column pair, token group)
    constexpr int CP = D / 2;
    constexpr int NTG = kAttnThreads / CP;
    const int cp = tid % CP, tg = tid / CP;
    float o[kGMax][2];
#pragma unroll
    for (int g = 0; g < kGMax; ++g) o[g][0] = o[g][1] = 0.0f;
    for (int t = tg; t < n; t += NTG) {
        const float2 v = __bfloat1622float2(
            *reinterpret_cast<const __nv_bfloat162*>(Vs + (size_t)t * D + 2 * cp));
#pragma unroll
        for (int g = 0; g < kGMax; ++g) {
            if (g < G) {
                const float pr = sc[g * chunk + t];
                o[g][0] = fmaf(pr, v.x, o[g][0]);
                o[g][1] = fmaf(pr, v.y, o[g][1]);
            }
        }
    }
    // Ks is no longer read: reuse it for the cross-group reduction
#pragma unroll
    for (int g = 0; g < kGMax; ++g) {
        if (g < G) {
            red[((size_t)tg * kGMax + g) * D + 2 * cp] = o[g][0];
            red[((size_t)tg * kGMax + g) * D + 2 * cp + 1] = o[g][1];
        }
    }
    attn_sync();
    for (int i = tid; i < G * D; i += kAttnThreads) {
        const int g = i / D, d = i - g * D;
        float acc = 0.0f;
#pragma unroll
        for (int q = 0; q < NTG; ++q) acc += red[((size_t)q * kGMax + g) * D + d];
        const int h = kvh * G + g;
        if (splits == 1) {
            const float val = n > 0 ? __fdiv_rn(acc, stat[2 * g + 1]) : 0.0f;
            p.out[((size_t)b * p.Hq + h) * D + d] = f2bf(val);
        } else {
            float* pp = p.part + (((size_t)b * p.Hq + h) * splits + split) * (D + 2);
            pp[d] = n > 0 ? acc : 0.0f;
            if (d == 0) {
                pp[D] = n > 0 ? stat[2 * g] : -INFINITY;
                pp[D + 1] = n > 0 ? stat[2 * g + 1] : 0.0f;
            }
        }
    }
    attn_sync();   // the shared tiles may be reused by the caller afterwards
}

// Combine of split-KV partials for (request b, query head h, element d).
template <int D>
__device__ __forceinline__ void attn_combine_elem(const float* part, int splits, int Hq, int b,
                                                  int h, int d, bf16* out) {
    const float* pp = part + ((size_t)b * Hq + h) * splits * (D + 2);
    float M = -INFINITY;
    for (int s = 0; s < splits; ++s) M = fmaxf(M, __ldcg(pp + (size_t)s * (D + 2) + D));
    float L = 0.0f, acc = 0.0f;
    if (M != -INFINITY) {
        for (int s = 0; s < splits; ++s) {
            const float m = __ldcg(pp + (size_t)s * (D + 2) + D);
            if (m == -INFINITY) continue;
            const float w = expf(m - M);
            L = fmaf(__ldcg(pp + (size_t)s * (D + 2) + D + 1), w, L);
            acc = fmaf(__ldcg(pp + (size_t)s * (D + 2) + d), w, acc);
        }
    }
    out[((size_t)b * Hq + h) * D + d] = f2bf(L > 0.0f ? __fdiv_rn(acc, L) : 0.0f);
}

}  // namespace a8w8
