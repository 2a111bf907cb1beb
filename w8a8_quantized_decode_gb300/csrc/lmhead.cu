// lmhead.cu -- standalone kernels of the decode step's ends (embedding
// gather, final RMSNorm + LM head + greedy argmax, device-side decode-loop
// advance) and the RoPE table; their device bodies live in lmhead_impl.cuh.
#include <algorithm>

#include "lmhead_impl.cuh"

namespace a8w8 {

namespace {

// 16 warps; weight ring of 8 batches of 2 steps (128 KB), 2 batches requested
// before the dependency wait; up to 8 batch rows per launch. The shared
// memory (at least kLmMinSmem) admits one CTA per SM: two CTAs sharing an SM
// would halve its share of the stream and leave the kernel waiting on that
// SM.
constexpr int kLmThreads = 512;
constexpr int kLmRingUnr = 2;
constexpr int kLmRingNB = 8;
constexpr size_t kLmMinSmem = 120 * 1024;
constexpr int kLmRingPre = 2;
constexpr int kLmMaxTile = 8;
constexpr size_t kLmRingBytes = lm::ring_bytes(kLmThreads, kLmRingUnr, kLmRingNB);

__global__ void embed_kernel(const bf16* __restrict__ embed, int vocab, int H,
                             const int32_t* __restrict__ ids, bf16* __restrict__ hidden,
                             unsigned long long* keys, unsigned* ticket, int B, unsigned* err) {
    pdl_wait();
    pdl_trigger();
    embed_rows(embed, vocab, H, ids, B, hidden, keys, ticket, err, blockIdx.x, gridDim.x);
}

__global__ void advance_kernel(int32_t* tok, int32_t* slot, const int32_t* table, int32_t* ctx,
                               const int32_t* next, int B, int max_blocks, int page) {
    pdl_wait();
    pdl_trigger();
    const int b = blockIdx.x * blockDim.x + threadIdx.x;
    if (b < B) advance_row(b, tok, slot, table, ctx, next, max_blocks, page);
}

__global__ void rope_table_kernel(float* rope, int D, double theta) {
    const int pos = blockIdx.x, i = threadIdx.x;
    const double inv_freq = pow(theta, -2.0 * (double)i / (double)D);
    const double ang = (double)pos * inv_freq;
    const double c = cos(ang), sn = sin(ang);
    const float ch = (float)c, sh = (float)sn;
    float* row = rope + (size_t)pos * 2 * D;
    row[i] = ch;
    row[D / 2 + i] = sh;
    row[D + i] = (float)(c - (double)ch);
    row[3 * D / 2 + i] = (float)(sn - (double)sh);
}

template <int BT>
__global__ void __launch_bounds__(kLmThreads, 1) lmhead_kernel(const LmHeadParams p) {
    extern __shared__ __align__(16) unsigned char smem[];
    lm::stream_lm<BT, kLmThreads, kLmRingUnr, kLmRingNB, kLmRingPre>(p, smem, [] {
        pdl_wait();
        pdl_trigger();
        return true;
    });
}

template <int BT>
cudaError_t launch_lm_t(const LmHeadParams& p, const Launch& L) {
    auto kern = lmhead_kernel<BT>;
    {
        // the shared-memory limit, set once per CUDA context
        cudaError_t e = once_per_context(reinterpret_cast<const void*>(kern), [&]() -> cudaError_t {
            cudaError_t e =
                cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
            return e;
        });
        if (e != cudaSuccess) return e;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(L.num_sms);
    cfg.blockDim = dim3(kLmThreads);
    cfg.dynamicSmemBytes = std::max(lm::smem_bytes(BT, p.H, kLmThreads, kLmRingBytes), kLmMinSmem);
    if (cfg.dynamicSmemBytes > 227 * 1024) return cudaErrorInvalidValue;
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
    if (p.M <= 8) return launch_lm_t<8>(p, L);
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
