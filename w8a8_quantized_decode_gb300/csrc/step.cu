// step.cu -- the whole decode step as one persistent cooperative kernel.
//
// One CTA per SM (512 threads) runs, in order: the embedding gather, for
// every layer the QKV projection (input RMSNorm + quantisation prologue), the
// fused QK-norm / RoPE / KV-write / paged attention, the O projection +
// residual, the Gate/Up projection + SwiGLU and the split-K down projection +
// residual, then the final RMSNorm + LM head + greedy argmax, and optionally
// the device-side decode-loop update. The per-op arithmetic is the same code
// as the standalone kernels (gemv_impl.cuh, attn_impl.cuh, lmhead_impl.cuh),
// so both paths give bit-identical results.
//
// Phases are separated by grid barriers. Before waiting at a barrier each CTA
// issues the first loads of its share of the next projection's weights (they
// never depend on the barrier), so HBM keeps streaming across phase
// boundaries and no kernel launch, ramp-up or tail separates the ~200 phases
// of a step. Every barrier wait is bounded: after ~2 s a CTA gives up, sets
// the timeout bit of the device error word and an abort flag that every other
// CTA checks, and all CTAs return; no launch can hang.
#include "attn_impl.cuh"
#include "gemv_impl.cuh"
#include "lmhead_impl.cuh"

namespace a8w8 {

namespace {

// 16 warps with a 128-register budget (64 registers per thread would spill
// inside the streaming loops of this much larger kernel), 4 units per batch.
constexpr int kStepThreads = 512;
constexpr unsigned long long kBarrierTimeoutNs = 2000000000ull;

__device__ __forceinline__ unsigned ld_acquire(const unsigned* p) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ unsigned long long global_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Grid-wide barrier number `k` (1, 2, ...): arrivals are counted on bar[0],
// which was zeroed before the launch, so barrier k completes at k * G.
// Returns false (in every thread of the CTA) if the step was aborted.
__device__ __forceinline__ bool grid_sync(unsigned* bar, unsigned* k, unsigned* err, int* s_ok) {
    __syncthreads();
    if (threadIdx.x == 0) {
        const unsigned kk = ++*k;
        const unsigned target = kk * gridDim.x;
        __threadfence();
        atomicAdd(&bar[0], 1u);
        int ok = 1;
        const unsigned long long t0 = global_ns();
        while (ld_acquire(&bar[0]) < target) {
            if (ld_acquire(&bar[1]) != 0u) {
                ok = 0;
                break;
            }
            if (global_ns() - t0 > kBarrierTimeoutNs) {
                atomicExch(&bar[1], 1u);
                set_error(err, 0x20u);
                ok = 0;
                break;
            }
            __nanosleep(64);
        }
        __threadfence();
        *s_ok = ok;
    }
    __syncthreads();
    return *s_ok != 0;
}

__device__ __forceinline__ void gemv_params(const StepParams& P, GemvParams& g) {
    g = GemvParams{};
    g.M = P.B;
    g.eps = P.eps;
    g.err = P.err;
}

// Weight ring of the projection phases: 2 units per batch, 6 batches (96 KB),
// 2 requested before the barrier.
constexpr int kStepRingUnr = 2;
constexpr int kStepRingNB = 6;
constexpr int kStepRingPre = 2;
constexpr size_t kStepRingBytes = gemv::ring_bytes<kStepThreads, kStepRingUnr, kStepRingNB>();

// One projection phase: issue the first weight loads of this CTA's share,
// wait for the producer of the activations (grid barrier), then stream.
template <int BT, int PRO, int EPI, int KS>
__device__ __forceinline__ bool gemv_phase(const GemvParams& g, unsigned char* smem, unsigned* bar,
                                           unsigned* k, unsigned* err, int* s_ok) {
    return gemv::stream_gemv<BT, PRO, EPI, KS, kStepThreads, kStepRingUnr, kStepRingNB, kStepRingPre>(
        g, smem, [&] { return grid_sync(bar, k, err, s_ok); });
}

template <int D>
__device__ __forceinline__ void attn_phase(const AttnParams& a, int chunk, int splits,
                                        unsigned char* smem) {
    const int items = a.B * a.Hq * splits;
    for (int it = blockIdx.x; it < items; it += gridDim.x) {
        const int split = it % splits;
        const int h = (it / splits) % a.Hq;
        const int b = it / (splits * a.Hq);
        attn_item<D, kStepThreads>(a, chunk, splits, split, h, b, smem, false);
    }
}

template <int BT>
__device__ __forceinline__ bool lm_phase(const LmHeadParams& lp, unsigned char* smem, unsigned* bar,
                                      unsigned* k, unsigned* err, int* s_ok, bool* last) {
    const int r = lm::stream_lm<BT, kStepThreads, kStepRingUnr, kStepRingNB, kStepRingPre>(
        lp, smem, [&] { return grid_sync(bar, k, err, s_ok); });
    *last = r == 1;
    return r >= 0;
}

template <int BT, int D, int KSD>
__global__ void __launch_bounds__(kStepThreads, 1) step_kernel(const __grid_constant__ StepParams P) {
    extern __shared__ __align__(16) unsigned char smem[];
    __shared__ int s_ok;
    __shared__ unsigned k;
    // Parameter blocks of the current phase, built by thread 0: the threads
    // read the fields from shared memory instead of holding them in registers.
    __shared__ GemvParams sg;
    __shared__ AttnParams sa;
    __shared__ LmHeadParams sl;
    const int cta = blockIdx.x, G = gridDim.x;
    const bool t0 = threadIdx.x == 0;
    if (t0) k = 0;
    const int NQ = P.Hq * P.D, NK = P.Hkv * P.D, NQKV = NQ + 2 * NK;
    const int max_ctx = P.max_blocks * P.page;
    const int chunk = max_ctx <= 256 ? 256 : 128;
    const int splits = (max_ctx + chunk - 1) / chunk;

    embed_rows(P.embed, P.vocab, P.H, P.token_ids, P.B, P.hidden, P.keys, P.ticket, P.err, cta, G);

    // Phases of a layer: 0 QKV, 1 attention, 2 O, 3 Gate/Up, 4 down. One switch
    // per phase keeps the register allocation of the phases separate.
    for (int ph = 0; ph < 5 * P.L; ++ph) {
        const int l = ph / 5, kind = ph - 5 * l;
        const StepLayer& W = P.layers[l];
        __syncthreads();   // every thread is done with the previous parameter block
        if (t0) {
            if (kind == 1) {
                AttnParams& a = sa;
                a = AttnParams{};
                a.q = P.qkv;
                a.q_stride = NQKV;
                a.fused = true;
                a.q_norm_w = W.q_norm_w;
                a.k_norm_w = W.k_norm_w;
                a.rope = P.rope;
                a.max_pos = P.max_pos;
                a.eps = P.eps;
                a.slot_mapping = P.slot_mapping;
                a.k_cache = P.k_cache[l];
                a.v_cache = P.v_cache[l];
                a.block_table = P.block_table;
                a.ctx_lens = P.ctx_lens;
                a.B = P.B;
                a.Hq = P.Hq;
                a.Hkv = P.Hkv;
                a.D = D;
                a.page = P.page;
                a.max_blocks = P.max_blocks;
                a.num_blocks = P.num_blocks;
                a.scale = P.attn_scale;
                a.scale_lo = P.attn_scale_lo;
                a.out = P.attn;
                a.part = P.part;
                a.err = P.err;
            } else {
                gemv_params(P, sg);
                if (kind == 0) {           // QKV with the input RMSNorm + quantisation prologue
                    sg.W = W.w_qkv;
                    sg.w_scale = W.s_qkv;
                    sg.K = P.H;
                    sg.N = NQKV;
                    sg.x = P.hidden;
                    sg.ldx = P.H;
                    sg.norm_w = W.input_norm_w;
                    sg.y = P.qkv;
                    sg.ldy = NQKV;
                } else if (kind == 2) {    // O + residual (quantisation prologue)
                    sg.W = W.w_o;
                    sg.w_scale = W.s_o;
                    sg.K = NQ;
                    sg.N = P.H;
                    sg.x = P.attn;
                    sg.ldx = NQ;
                    sg.residual = P.hidden;
                    sg.y = P.hidden;
                    sg.ldy = P.H;
                } else if (kind == 3) {    // Gate/Up + SwiGLU (post-attention RMSNorm prologue)
                    sg.W = W.w_gate_up;
                    sg.w_scale = W.s_gate_up;
                    sg.K = P.H;
                    sg.N = P.I;
                    sg.x = P.hidden;
                    sg.ldx = P.H;
                    sg.norm_w = W.post_norm_w;
                    sg.y = P.act;
                    sg.ldy = P.I;
                } else {                   // split-K down + residual (quantisation prologue)
                    sg.W = W.w_down;
                    sg.w_scale = W.s_down;
                    sg.K = P.I;
                    sg.N = P.H;
                    sg.x = P.act;
                    sg.ldx = P.I;
                    sg.residual = P.hidden;
                    sg.y = P.hidden;
                    sg.ldy = P.H;
                }
            }
        }
        __syncthreads();
        bool ok = true;
        switch (kind) {
            case 0:
                ok = gemv_phase<BT, PRO_NORM_QUANT, EPI_STORE, 1>(sg, smem, P.bar, &k, P.err, &s_ok);
                break;
            case 1:
                // QK norm, RoPE, KV write, paged attention (after the QKV results are complete)
                ok = grid_sync(P.bar, &k, P.err, &s_ok);
                if (ok) attn_phase<D>(sa, chunk, splits, smem);
                if (ok && splits > 1) {
                    ok = grid_sync(P.bar, &k, P.err, &s_ok);
                    if (ok) {
                        // one (request, query head) per CTA at a time: split
                        // weights by warp 0 (shared memory), then D elements
                        float* cw = reinterpret_cast<float*>(smem);
                        const int lane = threadIdx.x & 31;
                        for (int r = cta; r < P.B * P.Hq; r += G) {
                            const float* pp = P.part + (size_t)r * splits * (2 * D + 4);
                            __syncthreads();
                            if (threadIdx.x < 32) combine_weights<D>(pp, splits, cw, cw + 2 * splits, lane);
                            __syncthreads();
                            if ((int)threadIdx.x < D)
                                P.attn[(size_t)r * D + threadIdx.x] =
                                    combine_elem<D>(pp, splits, cw, cw + 2 * splits, threadIdx.x);
                        }
                    }
                }
                break;
            case 2:
                ok = gemv_phase<BT, PRO_QUANT, EPI_STORE, 1>(sg, smem, P.bar, &k, P.err, &s_ok);
                break;
            case 3:
                ok = gemv_phase<BT, PRO_NORM_QUANT, EPI_SWIGLU, 1>(sg, smem, P.bar, &k, P.err, &s_ok);
                break;
            default:
                ok = gemv_phase<BT, PRO_QUANT, EPI_STORE, KSD>(sg, smem, P.bar, &k, P.err, &s_ok);
                break;
        }
        if (!ok) return;
    }
    // final RMSNorm + LM head + greedy argmax
    {
        __syncthreads();
        if (t0) {
        LmHeadParams& lp = sl;
        lp = LmHeadParams{};
        lp.hidden = P.hidden;
        lp.norm_w = P.final_norm_w;
        lp.eps = P.eps;
        lp.W = P.lm_head;
        lp.H = P.H;
        lp.V = P.vocab;
        lp.M = P.B;
        lp.logits = P.logits;
        lp.final_hidden = P.final_hidden;
        lp.keys = P.keys;
        lp.ticket = P.ticket;
        lp.next_tokens = P.next_tokens;
        }
        __syncthreads();
        bool last = false;
        if (!lm_phase<BT>(sl, smem, P.bar, &k, P.err, &s_ok, &last)) return;
        if (last && P.device_loop && (int)threadIdx.x < P.B) {
            __threadfence();
            advance_row(threadIdx.x, P.token_ids, P.slot_mapping, P.block_table, P.ctx_lens,
                        P.next_tokens, P.max_blocks, P.page);
        }
    }
}

size_t step_smem_bytes(int BT, int D, int G, int H, int I, int Hq, int Hkv, int max_ctx, int ksd) {
    const int NQ = Hq * D, NQKV = NQ + 2 * Hkv * D;
    const size_t r = kStepRingBytes;
    size_t m = gemv::smem_layout(BT, 1, 1, H, NQKV, G, kStepThreads, r).total;
    m = std::max(m, gemv::smem_layout(BT, 1, 1, NQ, H, G, kStepThreads, r).total);
    m = std::max(m, gemv::smem_layout(BT, 2, 1, H, I, G, kStepThreads, r).total);
    m = std::max(m, gemv::smem_layout(BT, 1, ksd, I, H, G, kStepThreads, r).total);
    m = std::max(m, attn_item_smem_bytes(max_ctx <= 256 ? 256 : 128, D));
    m = std::max(m, lm::smem_bytes(BT, H, kStepThreads, lm::ring_bytes(kStepThreads, kStepRingUnr, kStepRingNB)));
    return m;
}

template <int BT, int D, int KSD>
cudaError_t launch_step_t(const StepParams& p, const Launch& L) {
    auto kern = step_kernel<BT, D, KSD>;
    const size_t smem = step_smem_bytes(BT, D, L.num_sms, p.H, p.I, p.Hq, p.Hkv,
                                        p.max_blocks * p.page, KSD);
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kStepThreads, smem);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) return cudaErrorCooperativeLaunchTooLarge;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(L.num_sms);
    cfg.blockDim = dim3(kStepThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = L.stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, p);
}

template <int BT>
cudaError_t launch_step_b(const StepParams& p, const Launch& L) {
    if (p.D != 128 || p.down_splits != 2) return cudaErrorInvalidValue;
    return launch_step_t<BT, 128, 2>(p, L);
}

}  // namespace

bool step_supported(int B, int D, int L, int H, int I, int Hq, int Hkv, int max_ctx, int num_sms) {
    // head_dim 128 with the two-way split-K down projection (the Qwen3-14B layer)
    if (B < 1 || B > 4 || L > kMaxStepLayers || D != 128) return false;
    const int NQ = Hq * D;
    // every projection must take the streaming path (K a multiple of 512 per split)
    if (H % 512 || NQ % 512 || I % 1024) return false;
    const int BT = B <= 1 ? 1 : B <= 2 ? 2 : 4;
    return step_smem_bytes(BT, D, num_sms, H, I, Hq, Hkv, max_ctx, 2) <= 227 * 1024;
}

cudaError_t launch_step(const StepParams& p, const Launch& L) {
    if (p.B <= 1) return launch_step_b<1>(p, L);
    if (p.B <= 2) return launch_step_b<2>(p, L);
    return launch_step_b<4>(p, L);
}

}  // namespace a8w8
