// gather.cu -- row gather for the prefill step: each sequence's last prompt
// row copied into a dense block, so that the final RMSNorm, LM head and
// argmax run on those rows only (the first generated token of each
// sequence).
#include "kernels.cuh"

namespace a8w8 {

namespace {

__global__ void __launch_bounds__(256) gather_rows_kernel(const bf16* __restrict__ src, int H,
                                                          const int32_t* __restrict__ rows,
                                                          int n_src, bf16* __restrict__ dst,
                                                          unsigned* err) {
    pdl_wait();
    pdl_trigger();
    const int s = blockIdx.x;
    const int r = rows[s];
    const bool ok = r >= 0 && r < n_src;
    if (!ok && threadIdx.x == 0) set_error(err, 0x40u);
    for (int i = threadIdx.x; i < H / 8; i += 256) {
        int4 v = make_int4(0, 0, 0, 0);
        if (ok) v = ld_cg_v4(src + (size_t)r * H + 8 * i);
        *reinterpret_cast<int4*>(dst + (size_t)s * H + 8 * i) = v;
    }
}

}  // namespace

cudaError_t launch_gather_rows(const bf16* src, int H, const int32_t* rows, int S, int n_src,
                               bf16* dst, unsigned* err, const Launch& L) {
    if (S <= 0) return cudaSuccess;
    if (H % 8) return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(S);
    cfg.blockDim = dim3(256);
    cfg.stream = L.stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = L.pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, gather_rows_kernel, src, H, rows, n_src, dst, err);
}

}  // namespace a8w8
