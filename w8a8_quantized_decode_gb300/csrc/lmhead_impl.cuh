// lmhead_impl.cuh -- device side of the decode step's ends: embedding gather,
// final RMSNorm + BF16 LM head + greedy argmax, and the device-side decode
// loop step; shared by the standalone kernels and the persistent step kernel.
//
// "Add Qwen3 A8W8 L2 runner foundation" (pypto-serving PR #61), "Related":
// embedding and sampling run on the device; "Add native Qwen3 14B A8W8
// serving path" (pypto-serving PR #48), "Performance" settings: temperature
// 0 and top_p 1, i.e. greedy decoding.
//
// LM head on the tensor cores (mma.sync m16n8k16, BF16 x BF16 -> FP32): the
// weight rows are the B operand (8 vocabulary rows per instruction), the
// normalised hidden rows the A operand (batch rows 0..7 of M = 16). CTA c
// owns 8-row groups [c*NG/G, (c+1)*NG/G); each warp owns whole groups and
// runs over all of K, so every logit is accumulated in one fixed order and is
// reproducible. Step s of a group: lane (g, c) = (lane / 4, lane % 4) copies
// the 16 bytes W[row0 + g][32 s + 8 c .. + 8) into its private slot of a
// cp.async shared-memory ring; its four BF16 pairs are the B fragments of
// two instructions, whose A fragments are the same eight columns of the
// hidden rows (the k order inside the 32 columns of a step is permuted
// identically on both sides, which leaves the dot products unchanged).
// FP32 logits; the argmax is reduced inside the CTA, merged across CTAs
// with a 64-bit atomic max on (order-preserving logit bits, inverted index)
// so ties go to the lowest index, and the last CTA to finish (atomic ticket,
// no waiting) writes the token ids and clears the keys.
#pragma once

#include "gemv_impl.cuh"

namespace a8w8 {
namespace lm {

__device__ __forceinline__ unsigned long long argmax_key(float v, int idx) {
    const unsigned u = __float_as_uint(v);
    const unsigned ord = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
    return ((unsigned long long)ord << 32) | (unsigned long long)(0xFFFFFFFFu - (unsigned)idx);
}

// Shared memory: hidden rows [BT][H + 32] BF16 (32 zero columns of padding
// keep the rows on different banks and cover a ragged last step), warp
// reductions, the weight ring.
__host__ __device__ constexpr size_t ring_bytes(int NT, int UNR, int NB) {
    return (size_t)NB * UNR * NT * 16;
}
__host__ __device__ inline size_t hn_stride(int H) { return (size_t)H + 32; }
__host__ __device__ inline size_t smem_bytes(int BT, int H, int nthreads, size_t ring) {
    const int nw = nthreads / 32;
    const size_t hn = ((size_t)BT * hn_stride(H) * 2 + 15) & ~size_t(15);
    const size_t red = (size_t)2 * gemv::kMaxWarps * BT * 4 + (size_t)nw * BT * 8 + 16;
    return ((hn + red + 127) & ~size_t(127)) + ring;
}

__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                               uint32_t a3, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
        "{%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// 16-byte cp.async that copies src_bytes (16 or 0) and zero-fills the rest,
// with an L2 cache policy.
__device__ __forceinline__ void cp_async16_zfill(uint32_t s, const void* g, int src_bytes,
                                                 uint64_t policy) {
    asm volatile("cp.async.cg.shared.global.L2::cache_hint [%0], [%1], 16, %2, %3;" ::"r"(s), "l"(g),
                 "r"(src_bytes), "l"(policy)
                 : "memory");
}

// One CTA's share of the LM head (BT <= 8 batch rows): NT threads, a weight
// ring of NB batches of UNR steps, NBPRE of them requested before `wait()`.
// Returns -1 if `wait` returned false, else 1 in the CTA that finished last
// (it wrote next_tokens) and 0 elsewhere.
template <int BT, int NT, int UNR, int NB, int NBPRE, class Wait>
__device__ __forceinline__ int stream_lm(const LmHeadParams& p, unsigned char* smem, Wait&& wait) {
    static_assert(BT <= 8, "the A operand holds batch rows 0..7");
    constexpr int NW = NT / 32;
    const int H = p.H, V = p.V, M = p.M;
    const int spr = (H + 31) / 32;          // steps per 8-row group
    const int NG = (V + 7) / 8;
    const int G = gridDim.x;
    const int cg0 = (int)(((long long)NG * blockIdx.x) / G);
    const int cg1 = (int)(((long long)NG * (blockIdx.x + 1)) / G);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int gr = lane >> 2, gc = lane & 3;
    const int wg0 = cg0 + (int)((long long)(cg1 - cg0) * warp / NW);
    const int wg1 = cg0 + (int)((long long)(cg1 - cg0) * (warp + 1) / NW);
    const int n = (wg1 - wg0) * spr;        // steps of this warp
    const bf16* W = p.W;

    const size_t hs = hn_stride(H);
    const size_t hn_bytes = ((size_t)BT * hs * 2 + 15) & ~size_t(15);
    bf16* hn = reinterpret_cast<bf16*>(smem);
    float* red = reinterpret_cast<float*>(smem + hn_bytes);          // [2 * kMaxWarps * BT]
    unsigned long long* best =
        reinterpret_cast<unsigned long long*>(red + 2 * gemv::kMaxWarps * BT);
    int* s_last = reinterpret_cast<int*>(best + NW * BT);
    const size_t ring_off =
        (hn_bytes + (size_t)2 * gemv::kMaxWarps * BT * 4 + (size_t)NW * BT * 8 + 16 + 127) & ~size_t(127);
    const uint32_t ring = (uint32_t)__cvta_generic_to_shared(smem + ring_off) + threadIdx.x * 16u;

    int lg = wg0, ls = 0, issued = 0;
    const uint64_t pol = l2_evict_first_policy();   // the LM head is streamed once per step
    auto issue_batch = [&](int slot) {
#pragma unroll
        for (int i = 0; i < UNR; ++i) {
            if (issued < n) {
                const int row = lg * 8 + gr, k = ls * 32 + 8 * gc;
                const bool ok = row < V && k < H;
                cp_async16_zfill(ring + (uint32_t)((slot * UNR + i) * NT * 16),
                                 ok ? (const void*)(W + (size_t)row * H + k) : (const void*)W,
                                 ok ? 16 : 0, pol);
                ++issued;
                if (++ls == spr) {
                    ls = 0;
                    ++lg;
                }
            }
        }
        cp_async_commit();
    };
#pragma unroll
    for (int b = 0; b < NBPRE; ++b) issue_batch(b);
    constexpr int NP = (8192 / 8 + NT - 1) / NT;   // RMSNorm weight (H <= 8192) in registers,
    int4 nwr[NP];                                   // loaded before the wait
    const int vec = H / 8;
    const bool nw_pre = vec <= NP * NT;
    if (nw_pre) {
#pragma unroll
        for (int i = 0; i < NP; ++i) {
            const int j = threadIdx.x + i * NT;
            nwr[i] = j < vec ? ld_nc_v4(p.norm_w + 8 * j) : make_int4(0, 0, 0, 0);
        }
    }

    if (!wait()) {
        cp_async_wait_all();
        return -1;
    }

    // final RMSNorm of the hidden rows (correctly rounded to BF16, see
    // norm_bf16): the raw rows are staged in hn, then normalised in place
    {
        f2 ss[BT];
#pragma unroll
        for (int b = 0; b < BT; ++b) ss[b].hi = ss[b].lo = 0.0f;
        for (int j = threadIdx.x; j < vec; j += NT) {
            int4 raw[BT];
#pragma unroll
            for (int b = 0; b < BT; ++b)
                raw[b] = b < M ? ld_cg_v4(p.hidden + (size_t)b * H + 8 * j) : make_int4(0, 0, 0, 0);
#pragma unroll
            for (int b = 0; b < BT; ++b) {
                *reinterpret_cast<int4*>(hn + (size_t)b * hs + 8 * j) = raw[b];
                float f[8];
                unpack8(raw[b], f);
#pragma unroll
                for (int e = 0; e < 8; ++e) f2_acc(ss[b], __fmul_rn(f[e], f[e]));
            }
        }
        // zero padding (a ragged last step multiplies it by zero weights)
        for (int i = threadIdx.x; i < BT * 32; i += NT)
            hn[(size_t)(i / 32) * hs + H + (i % 32)] = __float2bfloat16_rn(0.0f);
        // the rest of the ring, queued behind the hidden-row loads
#pragma unroll
        for (int b = NBPRE; b < NB; ++b) issue_batch(b);
        f2 inv[BT];
        gemv::block_rms_inv<BT>(ss, red, H, p.eps, inv);
        auto norm_vec = [&](int j, const int4 wraw) {
            float w[8];
            unpack8(wraw, w);
#pragma unroll
            for (int b = 0; b < BT; ++b) {
                float f[8];
                unpack8(*reinterpret_cast<const int4*>(hn + (size_t)b * hs + 8 * j), f);
                __align__(16) bf16 y[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) y[e] = norm_bf16(f[e], w[e], inv[b]);
                *reinterpret_cast<int4*>(hn + (size_t)b * hs + 8 * j) = *reinterpret_cast<const int4*>(y);
                if (blockIdx.x == 0 && p.final_hidden && b < M)
                    *reinterpret_cast<int4*>(p.final_hidden + (size_t)b * H + 8 * j) =
                        *reinterpret_cast<const int4*>(y);
            }
        };
        if (nw_pre) {
#pragma unroll
            for (int i = 0; i < NP; ++i) {
                const int j = threadIdx.x + i * NT;
                if (j < vec) norm_vec(j, nwr[i]);
            }
        } else {
            for (int j = threadIdx.x; j < vec; j += NT) norm_vec(j, ld_nc_v4(p.norm_w + 8 * j));
        }
        __syncthreads();
    }

    // A fragments come from hidden row gr (zero for rows >= M and for the
    // upper eight rows of the 16-row operand)
    const uint32_t hrow = (uint32_t)__cvta_generic_to_shared(hn) + (uint32_t)(gr * hs * 2) + 16u * gc;
    const bool arow = gr < M;
    float d[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    unsigned long long wbest = 0ull;          // this lane's best key for batch row gr
    int cgp = wg0, cs = 0, slot = 0;
    for (int done = 0; done < n; done += UNR) {
        cp_async_wait_group<NB - 1>();
        int4 w[UNR];
#pragma unroll
        for (int i = 0; i < UNR; ++i) w[i] = lds_v4(ring + (uint32_t)((slot * UNR + i) * NT * 16));
#pragma unroll
        for (int i = 0; i < UNR; ++i) {
            if (done + i < n) {
                int4 a = make_int4(0, 0, 0, 0);
                if (arow) a = lds_v4(hrow + (uint32_t)(cs * 64));
                mma_bf16_16816(d, (uint32_t)a.x, 0u, (uint32_t)a.y, 0u, (uint32_t)w[i].x, (uint32_t)w[i].y);
                mma_bf16_16816(d, (uint32_t)a.z, 0u, (uint32_t)a.w, 0u, (uint32_t)w[i].z, (uint32_t)w[i].w);
                if (++cs == spr) {
                    // d[0], d[1]: logits of batch row gr, vocabulary rows
                    // 8*cgp + 2*gc and + 1
                    const int row = cgp * 8 + 2 * gc;
                    if (arow) {
                        if (row < V) {
                            if (p.logits) p.logits[(size_t)gr * V + row] = d[0];
                            const unsigned long long k0 = argmax_key(d[0], row);
                            wbest = k0 > wbest ? k0 : wbest;
                        }
                        if (row + 1 < V) {
                            if (p.logits) p.logits[(size_t)gr * V + row + 1] = d[1];
                            const unsigned long long k1 = argmax_key(d[1], row + 1);
                            wbest = k1 > wbest ? k1 : wbest;
                        }
                    }
                    d[0] = d[1] = d[2] = d[3] = 0.0f;
                    cs = 0;
                    ++cgp;
                }
            }
        }
        issue_batch(slot);
        slot = slot + 1 == NB ? 0 : slot + 1;
    }
    cp_async_wait_all();
    // best key per batch row: over the four lanes of the row, then the warps
#pragma unroll
    for (int o = 1; o <= 2; o <<= 1) {
        const unsigned long long v = __shfl_xor_sync(0xffffffffu, wbest, o);
        wbest = v > wbest ? v : wbest;
    }
    if (gc == 0 && gr < BT) best[warp * BT + gr] = arow ? wbest : 0ull;
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
