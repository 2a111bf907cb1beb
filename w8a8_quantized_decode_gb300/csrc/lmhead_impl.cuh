// lmhead_impl.cuh -- device side of the decode step's ends: embedding gather,
// final RMSNorm + BF16 LM head + greedy argmax, and the device-side decode
// loop step; shared by the standalone kernels and the persistent step kernel.
//
// "Add Qwen3 A8W8 L2 runner foundation" (pypto-serving PR #61), "Related":
// embedding and sampling run on the device; "Add native Qwen3 14B A8W8
// serving path" (pypto-serving PR #48), "Performance" settings: temperature
// 0 and top_p 1, i.e. greedy decoding.
//
// LM head: CTA c owns vocabulary rows [cV/G, (c+1)V/G); each warp owns whole
// rows (so every logit is reduced in one fixed order and is reproducible) and
// streams them with double-buffered 128-bit L1-bypassing loads, 4 units of
// 512 bytes per batch; the first batch (and an L2 warm-up of the next units)
// is issued before the dependency wait. The hidden rows are read from L2
// once, staged in shared memory and normalised there. FP32 logits; the argmax is reduced inside the CTA, merged across CTAs
// with a 64-bit atomic max on (order-preserving logit bits, inverted index) so
// ties go to the lowest index, and the last CTA to finish (atomic ticket, no
// waiting) writes the token ids and clears the keys.
#pragma once

#include "kernels.cuh"

namespace a8w8 {
namespace lm {

constexpr int kUnit = 512;

__device__ __forceinline__ unsigned long long argmax_key(float v, int idx) {
    const unsigned u = __float_as_uint(v);
    const unsigned ord = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
    return ((unsigned long long)ord << 32) | (unsigned long long)(0xFFFFFFFFu - (unsigned)idx);
}

__host__ __device__ inline size_t smem_bytes(int BT, int H, int nthreads) {
    const int nw = nthreads / 32;
    return (size_t)BT * H * 4 + (size_t)nw * BT * 4 + (size_t)nw * BT * 8 + 16;
}

// One CTA's share of the LM head: NT threads, UNR units per batch. The first
// batch of weight loads and an L2 warm-up of the next `l2_ahead` units per
// warp are issued before `wait()`; returns -1 if `wait` returned false, else 1
// in the CTA that finished last (it wrote next_tokens) and 0 elsewhere.
template <int BT, int NT, int UNR, class Wait>
__device__ __forceinline__ int stream_lm(const LmHeadParams& p, unsigned char* smem, int l2_ahead,
                                         Wait&& wait) {
    constexpr int NW = NT / 32;
    const int H = p.H, V = p.V;
    const int row_bytes = H * 2;
    const int upr = (row_bytes + kUnit - 1) / kUnit;
    const int G = gridDim.x;
    const int r0 = (int)(((long long)V * blockIdx.x) / G);
    const int r1 = (int)(((long long)V * (blockIdx.x + 1)) / G);
    const int nrows = r1 - r0;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int wr0 = r0 + (int)((long long)nrows * warp / NW);
    const int wr1 = r0 + (int)((long long)nrows * (warp + 1) / NW);
    const int n = (wr1 - wr0) * upr;   // units of this warp
    const unsigned char* W = reinterpret_cast<const unsigned char*>(p.W);

    int lrow = 0, lch = 0;
    const unsigned char* lp = W + (size_t)wr0 * row_bytes + lane * 16;
    auto load_batch = [&](int4 (&dst)[UNR], int count) {
#pragma unroll
        for (int i = 0; i < UNR; ++i) {
            if (i < count) {
                dst[i] = make_int4(0, 0, 0, 0);
                if (lch * kUnit + lane * 16 < row_bytes) dst[i] = ld_stream_v4(lp);
                lp += kUnit;
                if (++lch == upr) {
                    lch = 0;
                    ++lrow;
                    lp = W + (size_t)(wr0 + lrow) * row_bytes + lane * 16;
                }
            }
        }
    };
    int4 wa[UNR], wb[UNR];
    load_batch(wa, n < UNR ? n : UNR);
    {
        const int m = n < UNR + l2_ahead ? n : UNR + l2_ahead;
        for (int base = UNR; base < m; base += 8) {
            const int u = base + (lane >> 2);
            if (u < m) {
                const int row = u / upr, ch = u - row * upr;
                const int off = ch * kUnit + (lane & 3) * 128;
                if (off < row_bytes) prefetch_line_l2(W + (size_t)(wr0 + row) * row_bytes + off);
            }
        }
    }

    if (!wait()) return -1;

    const int M = p.M;
    float* hn = reinterpret_cast<float*>(smem);                  // [BT][H]
    float* red = hn + (size_t)BT * H;                            // [NW][BT]
    unsigned long long* best = reinterpret_cast<unsigned long long*>(red + NW * BT);
    int* s_last = reinterpret_cast<int*>(best + NW * BT);

    // final RMSNorm of the hidden rows (float32, rounded to BF16)
    const int vec = H / 8;
    {
        float ss[BT];
#pragma unroll
        for (int b = 0; b < BT; ++b) ss[b] = 0.0f;
        for (int j = threadIdx.x; j < vec; j += NT) {
#pragma unroll
            for (int b = 0; b < BT; ++b) {
                if (b < M) {
                    const int4 raw = ld_cg_v4(p.hidden + (size_t)b * H + 8 * j);
                    float f[8];
                    unpack8(raw, f);
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        ss[b] += f[e] * f[e];
                        hn[(size_t)b * H + 8 * j + e] = f[e];   // staged raw row
                    }
                }
            }
        }
#pragma unroll
        for (int b = 0; b < BT; ++b) {
            const float t = warp_sum(ss[b]);
            if (lane == 0) red[warp * BT + b] = t;
        }
        __syncthreads();
        float inv[BT];
#pragma unroll
        for (int b = 0; b < BT; ++b) {
            float t = 0.0f;
            for (int w = 0; w < NW; ++w) t += red[w * BT + b];
            inv[b] = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(__fdiv_rn(t, (float)H), p.eps)));
        }
        for (int j = threadIdx.x; j < vec; j += NT) {
            float w[8];
            unpack8(ld_nc_v4(p.norm_w + 8 * j), w);
#pragma unroll
            for (int b = 0; b < BT; ++b) {
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const float f = b < M ? hn[(size_t)b * H + 8 * j + e] : 0.0f;
                    const bf16 y = f2bf(__fmul_rn(__fmul_rn(f, inv[b]), w[e]));
                    hn[(size_t)b * H + 8 * j + e] = bf2f(y);
                    if (blockIdx.x == 0 && p.final_hidden && b < M)
                        p.final_hidden[(size_t)b * H + 8 * j + e] = y;
                }
            }
        }
        __syncthreads();
    }

    float acc[BT];
    unsigned long long wbest[BT];
#pragma unroll
    for (int b = 0; b < BT; ++b) {
        wbest[b] = 0ull;
        acc[b] = 0.0f;
    }
    int cr = 0, cch = 0;
    auto compute_batch = [&](const int4 (&w)[UNR], int count) {
#pragma unroll
        for (int i = 0; i < UNR; ++i) {
            if (i < count) {
                const int off = cch * kUnit + lane * 16;
                if (off < row_bytes) {
                    float wf[8];
                    unpack8(w[i], wf);
                    const int k = off / 2;
#pragma unroll
                    for (int b = 0; b < BT; ++b) {
                        const float4 h0 = *reinterpret_cast<const float4*>(hn + (size_t)b * H + k);
                        const float4 h1 = *reinterpret_cast<const float4*>(hn + (size_t)b * H + k + 4);
                        float a = acc[b];
                        a = fmaf(wf[0], h0.x, a);
                        a = fmaf(wf[1], h0.y, a);
                        a = fmaf(wf[2], h0.z, a);
                        a = fmaf(wf[3], h0.w, a);
                        a = fmaf(wf[4], h1.x, a);
                        a = fmaf(wf[5], h1.y, a);
                        a = fmaf(wf[6], h1.z, a);
                        a = fmaf(wf[7], h1.w, a);
                        acc[b] = a;
                    }
                }
                if (++cch == upr) {
                    const int row = wr0 + cr;
#pragma unroll
                    for (int b = 0; b < BT; ++b) {
                        const float logit = warp_sum(acc[b]);
                        acc[b] = 0.0f;
                        if (lane == 0 && b < M) {
                            if (p.logits) p.logits[(size_t)b * V + row] = logit;
                            const unsigned long long key = argmax_key(logit, row);
                            wbest[b] = key > wbest[b] ? key : wbest[b];
                        }
                    }
                    cch = 0;
                    ++cr;
                }
            }
        }
    };
    int done = 0;
    while (done < n) {
        const int ca = n - done < UNR ? n - done : UNR;
        const int rest = n - done - ca;
        const int cb = rest < UNR ? rest : UNR;
        load_batch(wb, cb);
        compute_batch(wa, ca);
        done += ca;
        if (done >= n) break;
        const int rest2 = n - done - cb;
        const int ca2 = rest2 < UNR ? rest2 : UNR;
        load_batch(wa, ca2);
        compute_batch(wb, cb);
        done += cb;
    }

    if (lane == 0) {
#pragma unroll
        for (int b = 0; b < BT; ++b) best[warp * BT + b] = wbest[b];
    }
    __syncthreads();
    if ((int)threadIdx.x < M) {
        unsigned long long k = 0ull;
        for (int w = 0; w < NW; ++w) {
            const unsigned long long v = best[w * BT + threadIdx.x];
            k = v > k ? v : k;
        }
        atomicMax(&p.keys[threadIdx.x], k);
    }
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) *s_last = (atomicAdd(p.ticket, 1u) == gridDim.x - 1u);
    __syncthreads();
    const bool last = *s_last != 0;
    if (last) {
        __threadfence();
        if ((int)threadIdx.x < M) {
            const unsigned long long k = atomicExch(&p.keys[threadIdx.x], 0ull);
            p.next_tokens[threadIdx.x] = (int32_t)(0xFFFFFFFFu - (unsigned)(k & 0xFFFFFFFFull));
        }
        if (threadIdx.x == 0) *p.ticket = 0u;
    }
    return last ? 1 : 0;
}

}  // namespace lm

// Embedding rows of B tokens into hidden; rows are spread over the CTAs.
// The first CTA also clears the argmax keys and ticket of the step.
__device__ __forceinline__ void embed_rows(const bf16* embed, int vocab, int H, const int32_t* ids,
                                           int B, bf16* hidden, unsigned long long* keys,
                                           unsigned* ticket, unsigned* err, int cta, int G) {
    if (cta == 0) {
        for (int i = threadIdx.x; i < B; i += blockDim.x) keys[i] = 0ull;
        if (threadIdx.x == 0) *ticket = 0u;
    }
    const int vec = H / 8;
    for (int b = cta; b < B; b += G) {
        const int id = ids[b];
        const bool ok = id >= 0 && id < vocab;
        if (!ok && threadIdx.x == 0) set_error(err, 0x8u);
        for (int i = threadIdx.x; i < vec; i += blockDim.x) {
            int4 v = make_int4(0, 0, 0, 0);
            if (ok) v = ld_nc_v4(embed + (size_t)id * H + 8 * i);
            *reinterpret_cast<int4*>(hidden + (size_t)b * H + 8 * i) = v;
        }
    }
}

// Device-side decode loop: the next step's token ids are this step's argmax,
// the context grows by one token whose slot comes from the block table; a row
// whose context is full becomes a padded row. One thread per row.
__device__ __forceinline__ void advance_row(int b, int32_t* tok, int32_t* slot, const int32_t* table,
                                            int32_t* ctx, const int32_t* next, int max_blocks,
                                            int page) {
    const int c = ctx[b];
    if (c <= 0) {
        slot[b] = -1;
        return;
    }
    tok[b] = next[b];
    const int pos = c;   // position of the next token
    if (pos >= max_blocks * page) {
        ctx[b] = 0;
        slot[b] = -1;
        return;
    }
    ctx[b] = c + 1;
    slot[b] = table[(size_t)b * max_blocks + pos / page] * page + pos % page;
}

}  // namespace a8w8
