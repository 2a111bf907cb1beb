// attention.cu -- paged BF16 KV write and GQA decode attention (split-KV).
//
// "perf(qwen3-a8w8): optimize decode scheduling and data paths" (pypto-lib PR
// #810), "BF16 KV cache": K/V are stored in BF16 with no scale tensors and
// attention loads them directly; "Add Qwen3 A8W8 L2 runner foundation"
// (pypto-serving PR #61), "Summary": block table and slot mapping address the
// pages. "[Feature] Add native Qwen3-14B A8W8 serving path" (pypto-serving
// issue #52), "Current behavior": the decode layer normalises Q and K per head
// and applies RoPE before attention ("fused QK norm path").
//
// One CTA (256 threads) handles one (request, query head, token chunk); the
// device body and its arithmetic are described in attn_impl.cuh. Grid:
// (chunks, Hq, B). Decode layer: 64-token chunks (longer for contexts beyond
// 4096 tokens), only the chunks holding tokens run, and the last CTA of a
// (request, head) combines the partials (tickets in the workspace). The
// standalone entry uses 256/128-token chunks and a separate combine kernel
// (one CTA per query head and request).
#include "attn_impl.cuh"

namespace a8w8 {

// Contexts up to this length use the in-kernel combine in the decode layer.
constexpr int kInKernelMaxCtx = 64 * 256;
bool in_kernel_combine(int max_ctx, bool tickets) { return tickets && max_ctx <= kInKernelMaxCtx; }

namespace {

template <int D>
__global__ void __launch_bounds__(kAttnThreads) attn_kernel(const AttnParams p, int chunk,
                                                            int splits) {
    extern __shared__ __align__(16) unsigned char smem[];
    attn_item<D, kAttnThreads>(p, chunk, splits, blockIdx.x, blockIdx.y, blockIdx.z, smem, true);
}

// One CTA per (query head, request): split weights by warp 0 into shared
// memory, then one element per thread.
template <int D>
__global__ void __launch_bounds__(D) attn_combine_kernel(const float* __restrict__ part, int splits,
                                                         int Hq, bf16* __restrict__ out) {
    extern __shared__ float cws[];   // [splits][2] weights, then L[2]
    pdl_wait();
    pdl_trigger();
    const int h = blockIdx.x, b = blockIdx.y;
    const float* pp = part + ((size_t)b * Hq + h) * splits * (2 * D + 4);
    if (threadIdx.x < 32) combine_weights<D>(pp, splits, cws, cws + 2 * splits, threadIdx.x);
    __syncthreads();
    out[((size_t)b * Hq + h) * D + threadIdx.x] =
        combine_elem<D>(pp, splits, cws, cws + 2 * splits, threadIdx.x);
}

__global__ void kv_write_kernel(const bf16* __restrict__ k, const bf16* __restrict__ v, int T,
                                int row_vec, const int32_t* __restrict__ slot_mapping,
                                bf16* __restrict__ k_cache, bf16* __restrict__ v_cache,
                                long num_slots, unsigned* err) {
    pdl_wait();
    pdl_trigger();
    const long i = (long)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= (long)T * row_vec) return;
    const int t = (int)(i / row_vec), c = (int)(i - (long)t * row_vec);
    const long slot = slot_mapping[t];
    if (slot < 0) return;
    if (slot >= num_slots) {
        if (c == 0) set_error(err, 0x1u);
        return;
    }
    const int4 kv = ld_nc_v4(k + ((size_t)t * row_vec + c) * 8);
    const int4 vv = ld_nc_v4(v + ((size_t)t * row_vec + c) * 8);
    *reinterpret_cast<int4*>(k_cache + ((size_t)slot * row_vec + c) * 8) = kv;
    *reinterpret_cast<int4*>(v_cache + ((size_t)slot * row_vec + c) * 8) = vv;
}

template <typename Kern, typename... Args>
cudaError_t launch_ex(Kern kern, dim3 grid, dim3 block, size_t smem, const Launch& L,
                      Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = L.stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = L.pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kern, args...);
}

template <int D>
cudaError_t launch_attn_d(const AttnParams& p, const Launch& L) {
    const int max_ctx = p.max_blocks * p.page;
    const bool in_kernel = in_kernel_combine(max_ctx, p.tickets != nullptr);
    const int chunk = attn_chunk(max_ctx, in_kernel);
    const int splits = attn_splits(max_ctx, in_kernel);
    const size_t smem = attn_item_smem_bytes(chunk, D);
    {
        // the shared-memory limit, set once per CUDA context
        cudaError_t e = once_per_context(reinterpret_cast<const void*>(attn_kernel<D>), [&]() -> cudaError_t {
            cudaError_t e = cudaFuncSetAttribute(attn_kernel<D>,
                                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 (int)attn_item_smem_bytes(256, 128));
            return e;
        });
        if (e != cudaSuccess) return e;
    }
    AttnParams q = p;
    if (!in_kernel) q.tickets = nullptr;   // partials go to the combine kernel
    cudaError_t e = launch_ex(attn_kernel<D>, dim3(splits, p.Hq, p.B), dim3(kAttnThreads), smem,
                              L, q, chunk, splits);
    if (e != cudaSuccess || splits == 1 || in_kernel) return e;
    if ((size_t)(2 * splits + 2) * sizeof(float) > 48 * 1024) return cudaErrorInvalidValue;
    return launch_ex(attn_combine_kernel<D>, dim3(p.Hq, p.B), dim3(D),
                     (size_t)(2 * splits + 2) * sizeof(float), L, (const float*)p.part, splits, p.Hq,
                     p.out);
}

}  // namespace

// Standalone: one or two large chunks per CTA. In-kernel combine (decode
// layer, contexts up to kInKernelMaxCtx): chunks of 64 tokens, at most 64
// chunks per request (longer contexts get longer chunks, at most 256
// tokens); only the chunks that hold tokens run, and a context of one chunk
// needs no combine. Longer contexts use the standalone form.

int attn_chunk(int max_ctx, bool combine_in_kernel) {
    if (!in_kernel_combine(max_ctx, combine_in_kernel)) return max_ctx <= 256 ? 256 : 128;
    int c = (max_ctx + 63) / 64;
    c = (c + 15) / 16 * 16;
    return c < 64 ? 64 : (c > 256 ? 256 : c);
}

int attn_splits(int max_ctx, bool combine_in_kernel) {
    const int c = attn_chunk(max_ctx, combine_in_kernel);
    return max_ctx <= 0 ? 1 : (max_ctx + c - 1) / c;
}

size_t attn_part_bytes(int B, int Hq, int D, int max_ctx, bool combine_in_kernel) {
    const int s = attn_splits(max_ctx, combine_in_kernel);
    if (s <= 1) return 0;
    return (size_t)B * Hq * s * (2 * D + 4) * sizeof(float);
}

// Decode-layer attention over at least this many (request, cached token)
// slots of the launch shape uses the grouped form (attn_group.cu).
constexpr long kGroupMinWork = 8192;

cudaError_t launch_attention(const AttnParams& p, const Launch& L) {
    if (p.B == 0) return cudaSuccess;
    if ((long)p.B * p.max_blocks * p.page >= kGroupMinWork && attn_group_supported(p))
        return launch_attn_group(p, L);
    if (p.D == 128) return launch_attn_d<128>(p, L);
    if (p.D == 64) return launch_attn_d<64>(p, L);
    return cudaErrorInvalidValue;
}

cudaError_t launch_kv_write(const bf16* k, const bf16* v, int T, int Hkv, int D,
                            const int32_t* slot_mapping, bf16* k_cache, bf16* v_cache,
                            long num_slots, unsigned* err, const Launch& L) {
    if (T == 0) return cudaSuccess;
    const int row_vec = Hkv * D / 8;
    const long total = (long)T * row_vec;
    const int threads = 256;
    const int blocks = (int)((total + threads - 1) / threads);
    return launch_ex(kv_write_kernel, dim3(blocks), dim3(threads), 0, L, k, v, T, row_vec,
                     slot_mapping, k_cache, v_cache, num_slots, err);
}

}  // namespace a8w8
