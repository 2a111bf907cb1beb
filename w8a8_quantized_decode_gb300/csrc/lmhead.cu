// lmhead.cu -- embedding gather, RoPE table, final RMSNorm + BF16 LM head +
// greedy argmax.
//
// "Add Qwen3 A8W8 L2 runner foundation" (pypto-serving PR #61), "Related":
// embedding and sampling run on the device; "Add native Qwen3 14B A8W8
// serving path" (pypto-serving PR #48), "Performance" settings: temperature
// 0 and top_p 1, i.e. greedy decoding. The LM head streams its BF16 weights
// like the INT8 projections (one CTA per SM, whole rows per warp, 16-byte
// L1-bypassing loads, first loads issued before griddepcontrol.wait). The
// argmax is reduced inside each CTA, merged across CTAs with a 64-bit atomic
// max on (order-preserving logit bits, inverted index) so ties go to the
// lowest index, and the last CTA to finish (atomic ticket, no waiting) writes
// the token ids and clears the keys for the next step.
#include "kernels.cuh"

namespace a8w8 {

namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kUnit = 512;         // bytes per warp-wide load (256 BF16)
constexpr int kUnroll = 8;
constexpr int kLmMaxTile = 4;

__global__ void embed_kernel(const bf16* __restrict__ embed, int vocab, int H,
                             const int32_t* __restrict__ ids, bf16* __restrict__ hidden,
                             unsigned long long* keys, unsigned* ticket, int B, unsigned* err) {
    pdl_wait();
    pdl_trigger();
    const int b = blockIdx.x;
    if (b == 0) {
        for (int i = threadIdx.x; i < B; i += blockDim.x) keys[i] = 0ull;
        if (threadIdx.x == 0) *ticket = 0u;
    }
    const int id = ids[b];
    const bool ok = id >= 0 && id < vocab;
    if (!ok && threadIdx.x == 0) set_error(err, 0x8u);
    const int vec = H / 8;
    for (int i = threadIdx.x; i < vec; i += blockDim.x) {
        int4 v = make_int4(0, 0, 0, 0);
        if (ok) v = ld_nc_v4(embed + (size_t)id * H + 8 * i);
        *reinterpret_cast<int4*>(hidden + (size_t)b * H + 8 * i) = v;
    }
}

__global__ void advance_kernel(int32_t* tok, int32_t* slot, const int32_t* table, int32_t* ctx,
                               const int32_t* next, int B, int max_blocks, int page) {
    pdl_wait();
    pdl_trigger();
    const int b = blockIdx.x * blockDim.x + threadIdx.x;
    if (b >= B) return;
    const int c = ctx[b];
    if (c <= 0) {
        slot[b] = -1;
        return;
    }
    tok[b] = next[b];
    const int pos = c;   // position of the next token
    if (pos >= max_blocks * page) {
        ctx[b] = 0;      // context full: the row becomes padding
        slot[b] = -1;
        return;
    }
    ctx[b] = c + 1;
    slot[b] = table[(size_t)b * max_blocks + pos / page] * page + pos % page;
}

__global__ void rope_table_kernel(float* rope, int D, double theta) {
    const int pos = blockIdx.x, i = threadIdx.x;
    const double inv_freq = pow(theta, -2.0 * (double)i / (double)D);
    const double ang = (double)pos * inv_freq;
    rope[(size_t)pos * D + i] = (float)cos(ang);
    rope[(size_t)pos * D + D / 2 + i] = (float)sin(ang);
}

__device__ __forceinline__ unsigned long long argmax_key(float v, int idx) {
    const unsigned u = __float_as_uint(v);
    const unsigned ord = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
    return ((unsigned long long)ord << 32) | (unsigned long long)(0xFFFFFFFFu - (unsigned)idx);
}

template <int BT>
__global__ void __launch_bounds__(kThreads, 1) lmhead_kernel(const LmHeadParams p) {
    extern __shared__ __align__(16) unsigned char smem[];
    const int H = p.H, V = p.V, M = p.M;
    float* hn = reinterpret_cast<float*>(smem);                 // [BT][H]
    float* red = hn + (size_t)BT * H;                           // [kWarps][BT]
    unsigned long long* best = reinterpret_cast<unsigned long long*>(red + kWarps * BT);
    __shared__ int s_last;

    const int G = gridDim.x;
    const int r0 = (int)(((long long)V * blockIdx.x) / G);
    const int r1 = (int)(((long long)V * (blockIdx.x + 1)) / G);
    const int nrows = r1 - r0;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int wr0 = r0 + (int)((long long)nrows * warp / kWarps);
    const int wr1 = r0 + (int)((long long)nrows * (warp + 1) / kWarps);
    const int row_bytes = H * 2;
    const int upr = (row_bytes + kUnit - 1) / kUnit;
    const int U = (wr1 - wr0) * upr;
    const unsigned char* Wb = reinterpret_cast<const unsigned char*>(p.W);

    int lr = 0, lch = 0;
    int4 wv[kUnroll];
#pragma unroll
    for (int i = 0; i < kUnroll; ++i) {
        wv[i] = make_int4(0, 0, 0, 0);
        if (i < U) {
            const int off = lch * kUnit + lane * 16;
            if (off < row_bytes) wv[i] = ld_stream_v4(Wb + (size_t)(wr0 + lr) * row_bytes + off);
            if (++lch == upr) { lch = 0; ++lr; }
        }
    }

    pdl_wait();
    pdl_trigger();

    // final RMSNorm of the hidden rows (float32, rounded to BF16)
    const int vec = H / 8;
    {
        float ss[BT];
#pragma unroll
        for (int b = 0; b < BT; ++b) ss[b] = 0.0f;
        for (int j = threadIdx.x; j < vec; j += kThreads) {
#pragma unroll
            for (int b = 0; b < BT; ++b) {
                if (b < M) {
                    float f[8];
                    unpack8(ld_nc_v4(p.hidden + (size_t)b * H + 8 * j), f);
#pragma unroll
                    for (int e = 0; e < 8; ++e) ss[b] += f[e] * f[e];
                }
            }
        }
#pragma unroll
        for (int b = 0; b < BT; ++b) {
            const float s = warp_sum(ss[b]);
            if (lane == 0) red[warp * BT + b] = s;
        }
        __syncthreads();
        float inv[BT];
#pragma unroll
        for (int b = 0; b < BT; ++b) {
            float s = 0.0f;
#pragma unroll
            for (int w = 0; w < kWarps; ++w) s += red[w * BT + b];
            inv[b] = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(__fdiv_rn(s, (float)H), p.eps)));
        }
        for (int j = threadIdx.x; j < vec; j += kThreads) {
            float w[8];
            unpack8(ld_nc_v4(p.norm_w + 8 * j), w);
#pragma unroll
            for (int b = 0; b < BT; ++b) {
                float f[8];
                if (b < M) {
                    unpack8(ld_nc_v4(p.hidden + (size_t)b * H + 8 * j), f);
                } else {
#pragma unroll
                    for (int e = 0; e < 8; ++e) f[e] = 0.0f;
                }
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const bf16 y = f2bf(__fmul_rn(__fmul_rn(f[e], inv[b]), w[e]));
                    hn[(size_t)b * H + 8 * j + e] = bf2f(y);
                    if (blockIdx.x == 0 && p.final_hidden && b < M)
                        p.final_hidden[(size_t)b * H + 8 * j + e] = y;
                }
            }
        }
        __syncthreads();
    }

    unsigned long long wbest[BT];
#pragma unroll
    for (int b = 0; b < BT; ++b) wbest[b] = 0ull;
    float acc[BT];
#pragma unroll
    for (int b = 0; b < BT; ++b) acc[b] = 0.0f;
    int cr = 0, cch = 0;   // consume cursor (row offset within the warp's rows, chunk)
    for (int ub = 0; ub < U; ub += kUnroll) {
#pragma unroll
        for (int i = 0; i < kUnroll; ++i) {
            if (ub + i < U) {
                const int off = cch * kUnit + lane * 16;
                if (off < row_bytes) {
                    float wf[8];
                    unpack8(wv[i], wf);
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
        if (ub + kUnroll < U) {
#pragma unroll
            for (int i = 0; i < kUnroll; ++i) {
                if (ub + kUnroll + i < U) {
                    const int off = lch * kUnit + lane * 16;
                    wv[i] = make_int4(0, 0, 0, 0);
                    if (off < row_bytes)
                        wv[i] = ld_stream_v4(Wb + (size_t)(wr0 + lr) * row_bytes + off);
                    if (++lch == upr) { lch = 0; ++lr; }
                }
            }
        }
    }
    if (lane == 0) {
#pragma unroll
        for (int b = 0; b < BT; ++b) best[warp * BT + b] = wbest[b];
    }
    __syncthreads();
    if (threadIdx.x < M) {
        unsigned long long k = 0ull;
        for (int w = 0; w < kWarps; ++w) {
            const unsigned long long v = best[w * BT + threadIdx.x];
            k = v > k ? v : k;
        }
        atomicMax(&p.keys[threadIdx.x], k);
    }
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) s_last = (atomicAdd(p.ticket, 1u) == (unsigned)G - 1u);
    __syncthreads();
    if (s_last) {
        __threadfence();
        if (threadIdx.x < M) {
            const unsigned long long k = atomicExch(&p.keys[threadIdx.x], 0ull);
            p.next_tokens[threadIdx.x] = (int32_t)(0xFFFFFFFFu - (unsigned)(k & 0xFFFFFFFFull));
        }
        if (threadIdx.x == 0) *p.ticket = 0u;
    }
}

size_t lmhead_smem(int BT, int H) {
    return (size_t)BT * H * 4 + (size_t)kWarps * BT * 4 + (size_t)kWarps * BT * 8 + 16;
}

template <int BT>
cudaError_t launch_lm_t(const LmHeadParams& p, const Launch& L) {
    auto kern = lmhead_kernel<BT>;
    static int configured_dev = -1;
    int dev = 0;
    cudaGetDevice(&dev);
    if (configured_dev != dev) {
        cudaError_t e =
            cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024);
        if (e != cudaSuccess) return e;
        configured_dev = dev;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(L.num_sms);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = lmhead_smem(BT, p.H);
    cfg.stream = L.stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = L.pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kern, p);
}

}  // namespace

int lmhead_max_batch_tile() { return kLmMaxTile; }

cudaError_t launch_lmhead_argmax(const LmHeadParams& p, const Launch& L) {
    if (p.M <= 0) return cudaSuccess;
    if (p.M == 1) return launch_lm_t<1>(p, L);
    if (p.M == 2) return launch_lm_t<2>(p, L);
    if (p.M <= 4) return launch_lm_t<4>(p, L);
    return cudaErrorInvalidValue;
}

cudaError_t launch_embed(const bf16* embed, int vocab, int H, const int32_t* token_ids, int B,
                         bf16* hidden, unsigned long long* argmax_keys, unsigned* argmax_ticket,
                         unsigned* err, const Launch& L) {
    if (B == 0) return cudaSuccess;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(B);
    cfg.blockDim = dim3(256);
    cfg.stream = L.stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = L.pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, embed_kernel, embed, vocab, H, token_ids, hidden, argmax_keys,
                              argmax_ticket, B, err);
}

cudaError_t launch_advance(int32_t* token_ids, int32_t* slot_mapping, const int32_t* block_table,
                           int32_t* ctx_lens, const int32_t* next_tokens, int B, int max_blocks,
                           int page, const Launch& L) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((B + 63) / 64);
    cfg.blockDim = dim3(64);
    cfg.stream = L.stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = L.pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, advance_kernel, token_ids, slot_mapping, block_table, ctx_lens,
                              next_tokens, B, max_blocks, page);
}

cudaError_t launch_rope_table(float* rope, int max_pos, int D, double theta, cudaStream_t s) {
    if (max_pos == 0) return cudaSuccess;
    rope_table_kernel<<<max_pos, D / 2, 0, s>>>(rope, D, theta);
    return cudaGetLastError();
}

}  // namespace a8w8
