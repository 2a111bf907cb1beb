// quant.cu -- standalone per-row dynamic INT8 quantisation.
//
// "perf(qwen3-a8w8): optimize decode scheduling and data paths" (pypto-lib PR
// #810), "Decode scheduling" and "Gate/Up INT8 path": activations are
// quantised once per row, batched across decode rows. Per row: s = absmax /
// 127 and q = clamp(rne(x / s), -127, 127), both divisions IEEE float32.
// One CTA per row; the row is read twice (absmax, then codes), both passes
// with 16-byte loads. Inside the decode layer the same arithmetic runs as the
// prologue of each projection kernel instead.
#include "kernels.cuh"

namespace a8w8 {

namespace {

constexpr int kQuantThreads = 256;

__global__ void __launch_bounds__(kQuantThreads) quant_rows_kernel(const bf16* __restrict__ x,
                                                                   int cols, int ldx,
                                                                   int8_t* __restrict__ q,
                                                                   float* __restrict__ s) {
    pdl_wait();
    __shared__ float red[kQuantThreads / 32];
    const int row = blockIdx.x;
    const bf16* xr = x + (size_t)row * ldx;
    const int nvec = cols / 8;
    float amax = 0.0f;
    for (int i = threadIdx.x; i < nvec; i += kQuantThreads) {
        float f[8];
        unpack8(ld_nc_v4(xr + 8 * i), f);
#pragma unroll
        for (int j = 0; j < 8; ++j) amax = fmaxf(amax, fabsf(f[j]));
    }
    amax = warp_max(amax);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = amax;
    __syncthreads();
    if (threadIdx.x < 32) {
        float v = threadIdx.x < kQuantThreads / 32 ? red[threadIdx.x] : 0.0f;
        v = warp_max(v);
        if (threadIdx.x == 0) red[0] = v;
    }
    __syncthreads();
    const float sc = __fdiv_rn(red[0], 127.0f);
    const float rc = quant_recip(sc);
    if (threadIdx.x == 0) s[row] = sc;
    int8_t* qr = q + (size_t)row * cols;
    for (int i = threadIdx.x; i < nvec; i += kQuantThreads) {
        float f[8];
        unpack8(ld_nc_v4(xr + 8 * i), f);
        uint32_t lo = 0, hi = 0;
#pragma unroll
        for (int j = 0; j < 4; ++j) lo |= (uint32_t)(quant_code(f[j], sc, rc) & 0xff) << (8 * j);
#pragma unroll
        for (int j = 0; j < 4; ++j) hi |= (uint32_t)(quant_code(f[4 + j], sc, rc) & 0xff) << (8 * j);
        *reinterpret_cast<uint2*>(qr + 8 * i) = make_uint2(lo, hi);
    }
}

}  // namespace

cudaError_t launch_quant_rows(const bf16* x, int rows, int cols, int ldx, int8_t* q, float* s,
                              const Launch& L) {
    if (rows == 0) return cudaSuccess;
    quant_rows_kernel<<<rows, kQuantThreads, 0, L.stream>>>(x, cols, ldx, q, s);
    return cudaGetLastError();
}

}  // namespace a8w8
