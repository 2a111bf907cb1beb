// lmhead.cu -- standalone kernels of the decode step's ends (embedding
// gather, final RMSNorm + LM head + greedy argmax, device-side decode-loop
// advance) and the RoPE table; their device bodies live in lmhead_impl.cuh.
#include "lmhead_impl.cuh"

namespace a8w8 {

namespace {

// 32 warps for one row; 16 warps (more registers each) for 2-4 rows.
__host__ __device__ constexpr int lm_threads(int BT) { return BT >= 2 ? 512 : 1024; }
constexpr int kLmMaxTile = 4;
// Units per warp fetched into L2 before the dependency wait.
constexpr int kLmL2Ahead = 4;

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
    rope[(size_t)pos * D + i] = (float)cos(ang);
    rope[(size_t)pos * D + D / 2 + i] = (float)sin(ang);
}

template <int BT>
__global__ void __launch_bounds__(lm_threads(BT), 1) lmhead_kernel(const LmHeadParams p) {
    extern __shared__ __align__(16) unsigned char smem[];
    lm::stream_lm<BT, lm_threads(BT), 4>(p, smem, kLmL2Ahead, [] {
        pdl_wait();
        pdl_trigger();
        return true;
    });
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
    cfg.blockDim = dim3(lm_threads(BT));
    cfg.dynamicSmemBytes = lm::smem_bytes(BT, p.H, lm_threads(BT));
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
