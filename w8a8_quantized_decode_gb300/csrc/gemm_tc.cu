// gemm_tc.cu -- INT8 x INT8 -> INT32 projections of a prefill chunk on the
// fifth-generation tensor cores (tcgen05, accumulators in tensor memory).
//
// Arithmetic ("perf(qwen3-a8w8): optimize decode scheduling and data paths",
// pypto-lib PR #810, "Gate/Up INT8 path": INT8 x INT8 products accumulated
// exactly, dequantised in FP32 afterwards): C[m][n] = sum_{k in [k0, k1)}
// X[m][k] * W[n][k], X the INT8 activation codes [M, K], W the INT8 weights
// [N, K]. sm_103a has no INT8 kind of tcgen05.mma, so each code is fed as its
// FP16 image (exact: |code| <= 128 needs 8 significant bits) to the kind::f16
// MMA with FP32 accumulators. Every product is an integer of magnitude below
// 2^14 and 1024 of them sum to below 2^24, where FP32 holds every integer, so
// each 1024-column chunk of K accumulates exactly; the chunk's FP32 result is
// converted to INT32 and added to an INT32 running sum.
//
// One CTA computes a 128 x 256 tile of C^T (128 weight rows = the MMA's M and
// the tensor-memory lanes, 256 activation rows = the MMA's N and columns)
// over K steps of 64 columns. The activation codes arrive as their FP16
// images (i8_to_f16_kernel, once per projection), so TMA stores that operand
// directly in the 128-byte swizzled K-major layout the MMA reads; only the
// weight tile is converted in the kernel. (An m128 n256 k16 MMA does twice the
// work of an m128 n128 one in about 1.3x the time on this GPU, so the wider
// tile is the one that approaches the tensor peak.) Warp roles:
//   warp 0      TMA: per step the X tile (256 rows x 64 FP16, 32 KB, swizzled)
//               and the W tile (128 x 64 INT8, 8 KB) into a 4-stage ring; a
//               stage is reused once the MMAs of its pair of steps are done;
//   warp 1      allocates 512 tensor-memory columns; one thread issues the
//               MMAs (four per step) and commits once per pair of steps (a
//               commit costs the issuing thread about as much as three MMAs);
//   warps 2-9   convert the W tiles to FP16 in the swizzled layout, in two
//               groups of 4 warps that take alternate pairs of steps, each
//               into its own slot of two tiles;
//   warps 10-17 drain each finished chunk: the FP32 accumulators (256
//               columns, one buffer: the next chunk's first MMA waits for the
//               drain) to INT32, added into a 256-column INT32 sum in tensor
//               memory; after the last chunk they write C. Two warps per lane
//               quarter, 128 columns each.
// Every wait is bounded (2 s): on a timeout the CTA sets the device error
// word's timeout bit, every role stops, the in-flight copies and MMAs are
// waited for (again bounded) and the tensor memory is freed.
#include <cuda.h>

#include <algorithm>

#include "kernels.cuh"
#include "tc_common.cuh"

namespace a8w8 {

namespace {

using namespace tc;

constexpr int kTM = 128;          // weight rows per tile (the MMA's M)
constexpr int kTN = 256;          // activation rows per tile (the MMA's N)
constexpr int kTK = 64;           // K columns per step
constexpr int kChunkSteps = 16;   // steps per exact FP32 chunk (1024 columns)
constexpr int kStages8 = 4;       // TMA stages (X FP16 tile + W INT8 tile), two pairs of steps
constexpr int kStages16 = 4;      // converted W tiles: one slot of two per converter group
constexpr int kConvGroups = 2;    // converter groups of 4 warps, alternating pairs of steps
constexpr int kDrainWarps = 8;    // two per tensor-memory lane quarter, 128 columns each
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kSumCol = 256;  // INT32 sums at columns [256, 512); FP32 chunk at [0, 256)
constexpr int kTileW8 = kTM * kTK;           // 8192 bytes
constexpr int kTileW16 = kTM * kTK * 2;      // 16384 bytes
constexpr int kTileX16 = kTN * kTK * 2;      // 32768 bytes

struct TcSmem {
    size_t x16, w16, w8, bars, total;
};
// kS8 TMA stages, kS16 converted W tiles
template <int kS8, int kS16>
__host__ __device__ constexpr TcSmem tc_smem() {
    TcSmem s{};
    s.x16 = 0;                                        // [kS8][32 KB], 1024-aligned, TMA-swizzled
    s.w16 = s.x16 + (size_t)kS8 * kTileX16;           // [kS16][16 KB], 1024-aligned
    s.w8 = s.w16 + (size_t)kS16 * kTileW16;           // [kS8][8 KB]
    s.bars = s.w8 + (size_t)kS8 * kTileW8;
    // barriers: full8, empty8 [kS8]; full16 [kS16]; empty16 [kConvGroups];
    // accfull, accempty; done; then the tensor-memory base and the abort flag
    s.total = s.bars + (size_t)(2 * kS8 + kS16 + kConvGroups + 2 + 1) * 8 + 16;
    return s;
}
// dynamic shared memory requested: the layout plus room to align it to 1024
template <int kS8, int kS16>
constexpr size_t tc_smem_bytes() { return tc_smem<kS8, kS16>().total + 1024; }

// 16 INT8 codes -> 16 FP16 values (exact): byte v becomes the FP16 number
// 1024 + (v + 128), from which 1152 is subtracted.
__device__ __forceinline__ void i8x4_to_f16x4(uint32_t w, uint32_t& lo, uint32_t& hi) {
    const uint32_t u = w ^ 0x80808080u;
    const uint32_t l = __byte_perm(u, 0x64646464u, 0x4140);
    const uint32_t h = __byte_perm(u, 0x64646464u, 0x4342);
    const __half2 off = __halves2half2(__ushort_as_half(0x6480), __ushort_as_half(0x6480));
    const __half2 lf = __hsub2(*reinterpret_cast<const __half2*>(&l), off);
    const __half2 hf = __hsub2(*reinterpret_cast<const __half2*>(&h), off);
    lo = *reinterpret_cast<const uint32_t*>(&lf);
    hi = *reinterpret_cast<const uint32_t*>(&hf);
}

// Converts one 128 x 64 INT8 tile (row pitch 64 bytes) into the FP16
// 128-byte-swizzled K-major tile, thread t of 128 taking the 16-byte pieces
// t, t + 128, t + 256, t + 384 (piece p: row p / 4, columns 16 (p % 4) ..).
// All four pieces are loaded before any is converted.
__device__ __forceinline__ void convert_tile(const int8_t* src, unsigned char* dst, int t) {
    int4 vs[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int p = t + 128 * i;
        vs[i] = *reinterpret_cast<const int4*>(src + (p >> 2) * kTK + 16 * (p & 3));
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int p = t + 128 * i;
        const int r = p >> 2, q = p & 3;
        const int4 v = vs[i];
        uint4 a, b;
        i8x4_to_f16x4((uint32_t)v.x, a.x, a.y);
        i8x4_to_f16x4((uint32_t)v.y, a.z, a.w);
        i8x4_to_f16x4((uint32_t)v.z, b.x, b.y);
        i8x4_to_f16x4((uint32_t)v.w, b.z, b.w);
        // FP16 chunks 2q and 2q + 1 of row r, swizzled within the 8-row atom
        unsigned char* row = dst + (r >> 3) * 1024 + (r & 7) * 128;
        *reinterpret_cast<uint4*>(row + (((2 * q) ^ (r & 7)) << 4)) = a;
        *reinterpret_cast<uint4*>(row + (((2 * q + 1) ^ (r & 7)) << 4)) = b;
    }
}

// The timeout bit of the device error word (A8W8_DEVERR_TIMEOUT).
constexpr unsigned kErrTimeout = 0x20u;

__device__ __forceinline__ void set_timeout(unsigned* err, volatile int* abort) {
    *abort = 1;
    set_error(err, kErrTimeout);
}

}  // namespace

namespace {

// warps: TMA, MMA, 2 groups of 4 converter warps, 8 drain warps
constexpr int kTcThreads = (2 + 4 * kConvGroups + kDrainWarps) * 32;

template <int kS8, int kS16>
__global__ void __launch_bounds__(kTcThreads, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap map_w, const __grid_constant__ CUtensorMap map_x,
                   int M, int N, int k0, int steps, int32_t* __restrict__ C, int ldc,
                   unsigned* err) {
    static_assert(kS8 == 2 * kConvGroups && kS16 == 2 * kConvGroups && kConvGroups == 2,
                  "a TMA pair of stages and a converted slot per pair of steps");
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    // the swizzled tiles need 1024-byte aligned bases
    unsigned char* smem = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    constexpr TcSmem L = tc_smem<kS8, kS16>();
    unsigned char* x16 = smem + L.x16;
    unsigned char* w16 = smem + L.w16;
    int8_t* w8 = reinterpret_cast<int8_t*>(smem + L.w8);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L.bars);
    uint64_t* full8 = bars;                   // TMA stage landed
    uint64_t* empty8 = full8 + kS8;           // MMAs of the stage's step done
    uint64_t* full16 = empty8 + kS8;          // converted W tile written
    uint64_t* empty16 = full16 + kS16;        // MMAs of the slot's pair done
    uint64_t* accfull = empty16 + kConvGroups;
    uint64_t* accempty = accfull + 1;
    uint64_t* done = accempty + 1;
    uint32_t* tmem_base_smem = reinterpret_cast<uint32_t*>(done + 1);
    volatile int* abort = reinterpret_cast<volatile int*>(tmem_base_smem + 1);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int m0 = blockIdx.x * kTN;      // activation rows of the tile
    const int n0 = blockIdx.y * kTM;      // weight rows of the tile
    const int npairs = (steps + 1) / 2;
    const int nchunks = (steps + kChunkSteps - 1) / kChunkSteps;

    if (tid == 0) {
        for (int i = 0; i < kS8; ++i) {
            mbar_init(&full8[i], 1);      // the producer's expect-tx arrival
            mbar_init(&empty8[i], 1);     // the MMA commit
        }
        for (int i = 0; i < kS16; ++i) mbar_init(&full16[i], 4);   // one per converter warp
        for (int i = 0; i < kConvGroups; ++i) mbar_init(&empty16[i], 1);   // the MMA commit
        mbar_init(accfull, 1);            // the MMA commit
        mbar_init(accempty, kDrainWarps); // one arrival per drain warp
        mbar_init(done, 1);
        *abort = 0;
        mbar_init_fence();
        tma_prefetch_map(&map_w);
        tma_prefetch_map(&map_x);
    }
    if (warp == 1) tmem_alloc(tmem_base_smem, kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_base_smem;

    // the activation images come from the preceding kernel
    pdl_wait();
    pdl_trigger();

    if (warp == 0) {
        // ---- TMA producer: step s into stage s % kS8, once the MMAs of step
        // s - kS8 are done ----
        int issued = 0;
        if (lane == 0) {
            for (int s = 0; s < steps; ++s) {
                const int st = s % kS8;
                if (s >= kS8 && !mbar_wait(&empty8[st], ((s / kS8) - 1) & 1, abort)) {
                    if (!*abort) set_timeout(err, abort);
                    break;
                }
                mbar_arrive_expect_tx(&full8[st], kTileX16 + kTileW8);
                tma_load_2d(x16 + (size_t)st * kTileX16, &map_x, k0 + s * kTK, m0, &full8[st]);
                tma_load_2d(w8 + (size_t)st * kTileW8, &map_w, k0 + s * kTK, n0, &full8[st]);
                issued = s + 1;
            }
            // every issued copy has landed before the CTA may exit (immediate
            // on the normal path, where the MMAs consumed them all)
            for (int s = issued > kS8 ? issued - kS8 : 0; s < issued; ++s)
                mbar_wait(&full8[s % kS8], (s / kS8) & 1, nullptr);
        }
    } else if (warp == 1) {
        // ---- MMA issuer: A = converted W tile, B = X tile as TMA stored it ----
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_f16_f32(kTM, kTN);
            bool ok = true;
            for (int P = 0; P < npairs && ok; ++P) {
                const int s0 = 2 * P, ns = min(2, steps - s0);
                const int c = s0 / kChunkSteps;
                const bool first = s0 % kChunkSteps == 0;
                // a chunk's first MMA overwrites the FP32 accumulators: the
                // drain of the previous chunk must have read them
                if (first && c >= 1) ok = mbar_wait(accempty, (c - 1) & 1, abort);
                const int slot = P % kConvGroups;
                for (int u = 0; u < ns && ok; ++u) {
                    ok = mbar_wait(&full16[2 * slot + u], (P / kConvGroups) & 1, abort) &&
                         mbar_wait(&full8[(s0 + u) % kS8], ((s0 + u) / kS8) & 1, abort);
                    if (!ok) break;
                    tc_fence_after();
                    const uint64_t ad =
                        sw128_kmajor_desc(smem_u32(w16 + (size_t)(2 * slot + u) * kTileW16));
                    const uint64_t bd =
                        sw128_kmajor_desc(smem_u32(x16 + (size_t)((s0 + u) % kS8) * kTileX16));
#pragma unroll
                    for (int j = 0; j < kTK / 16; ++j)
                        mma_f16(tmem, ad + 2 * j, bd + 2 * j, idesc,
                                (first && u == 0 && j == 0) ? 0u : 1u);
                    // the TMA stage is free once this step's MMAs are done
                    mma_commit(&empty8[(s0 + u) % kS8]);
                }
                if (!ok) {
                    if (!*abort) set_timeout(err, abort);
                    break;
                }
                // the converted slot is free once the pair's MMAs are done
                mma_commit(&empty16[slot]);
                const int s1 = s0 + ns - 1;
                if (s1 % kChunkSteps == kChunkSteps - 1 || s1 == steps - 1) mma_commit(accfull);
            }
            // no MMA may still be running when the tensor memory is freed
            mma_commit(done);
            mbar_wait(done, 0, nullptr);
        }
    } else if (warp < 2 + 4 * kConvGroups) {
        // ---- converters: W INT8 tiles -> FP16 swizzled tiles; group g of 4
        // warps takes the step pairs P = g (mod 2) into its slot (tiles 2g,
        // 2g + 1) ----
        const int grp = (warp - 2) >> 2;
        const int t = tid - 64 - 128 * grp;
        for (int P = grp; P < npairs; P += kConvGroups) {
            const int s0 = 2 * P, ns = min(2, steps - s0), use = P / kConvGroups;
            bool ok = use == 0 || mbar_wait(&empty16[grp], (use - 1) & 1, abort);
            for (int u = 0; u < ns && ok; ++u) {
                ok = mbar_wait(&full8[(s0 + u) % kS8], ((s0 + u) / kS8) & 1, abort);
                if (!ok) break;
                convert_tile(w8 + (size_t)((s0 + u) % kS8) * kTileW8,
                             w16 + (size_t)(2 * grp + u) * kTileW16, t);
                fence_async_shared();
                __syncwarp();
                if (lane == 0) mbar_arrive(&full16[2 * grp + u]);
            }
            if (!ok) {
                if (!*abort) set_timeout(err, abort);
                break;
            }
        }
    } else {
        // ---- drain: FP32 chunk -> INT32 sum; after the last chunk, C. Warp
        // w takes lane quarter w % 4 and columns [128 h, 128 h + 128) ----
        const int q = warp & 3;
        const int h = (warp - 2 - 4 * kConvGroups) >> 2;
        const uint32_t lane_base = tmem + ((uint32_t)(32 * q) << 16);
        const int n = n0 + 32 * q + lane;             // this thread's weight row
        for (int c = 0; c < nchunks; ++c) {
            if (!mbar_wait(accfull, c & 1, abort)) {
                if (!*abort) set_timeout(err, abort);
                break;
            }
            tc_fence_after();
            const bool last = c == nchunks - 1;
#pragma unroll 1
            for (int g = 0; g < 4; ++g) {
                const uint32_t col = (uint32_t)(128 * h + 32 * g);
                uint32_t f[32], a[32];
                if (c > 0) {
                    tmem_ld32x2(lane_base + col, f, lane_base + kSumCol + col, a);
                } else {
                    tmem_ld32(lane_base + col, f);
#pragma unroll
                    for (int i = 0; i < 32; ++i) a[i] = 0u;
                }
#pragma unroll
                for (int i = 0; i < 32; ++i)
                    a[i] = (uint32_t)((int)a[i] + __float2int_rn(__uint_as_float(f[i])));
                if (!last) {
                    tmem_st32(lane_base + kSumCol + col, a);
                } else if (n < N) {
                    // C[m][n]: for each column the warp's lanes write 32
                    // consecutive words
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        const int m = m0 + (int)col + i;
                        if (m < M) C[(size_t)m * ldc + n] = (int32_t)a[i];
                    }
                }
            }
            if (!last) {
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(accempty);
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) {
        __syncwarp();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// Driver entry point that encodes tensor maps (resolved once per process).
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_tiled() {
    static EncodeTiledFn fn = [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                             &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return static_cast<EncodeTiledFn>(nullptr);
        return reinterpret_cast<EncodeTiledFn>(f);
    }();
    return fn;
}

// Tensor map of an INT8 matrix [rows, cols] (row pitch `ld` bytes) read in
// boxes of 128 rows x 64 bytes, zero-filled beyond the matrix.
bool make_i8_map(CUtensorMap* map, const int8_t* base, int rows, int cols, int ld) {
    EncodeTiledFn enc = encode_tiled();
    if (!enc) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)ld};
    const cuuint32_t box[2] = {(cuuint32_t)kTK, 128u};
    const cuuint32_t estr[2] = {1u, 1u};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<int8_t*>(base), dims, strides, box,
               estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Tensor map of an FP16 matrix [rows, cols] (row pitch 2 cols bytes) read in
// boxes of 256 rows x 64 values (128 bytes) and stored in the 128-byte
// swizzle, which is the K-major layout the MMA reads; zero-filled beyond the
// matrix.
bool make_f16_map(CUtensorMap* map, const uint16_t* base, int rows, int cols) {
    EncodeTiledFn enc = encode_tiled();
    if (!enc) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
    const cuuint32_t box[2] = {(cuuint32_t)kTK, (cuuint32_t)kTN};
    const cuuint32_t estr[2] = {1u, 1u};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<uint16_t*>(base), dims, strides,
               box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// FP16 images of INT8 codes (exact), 16 codes per thread.
__global__ void i8_to_f16_kernel(const int8_t* __restrict__ x, size_t n16, uint16_t* __restrict__ y) {
    pdl_wait();
    pdl_trigger();
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n16;
         i += (size_t)gridDim.x * blockDim.x) {
        const int4 v = __ldcs(reinterpret_cast<const int4*>(x) + i);
        uint4 a, b;
        i8x4_to_f16x4((uint32_t)v.x, a.x, a.y);
        i8x4_to_f16x4((uint32_t)v.y, a.z, a.w);
        i8x4_to_f16x4((uint32_t)v.z, b.x, b.y);
        i8x4_to_f16x4((uint32_t)v.w, b.z, b.w);
        reinterpret_cast<uint4*>(y)[2 * i] = a;
        reinterpret_cast<uint4*>(y)[2 * i + 1] = b;
    }
}

template <int kS8, int kS16>
cudaError_t launch_tc_t(const CUtensorMap& mw, const CUtensorMap& mx, int M, int N, int k0, int steps,
                        int32_t* C, int ldc, unsigned* err, const Launch& L) {
    auto kern = gemm_tc_kernel<kS8, kS16>;
    constexpr size_t smem = tc_smem_bytes<kS8, kS16>();
    static_assert(smem <= 227 * 1024, "shared memory");
    {
        // the shared-memory limit, set once per CUDA context
        cudaError_t e = once_per_context(reinterpret_cast<const void*>(kern), [&]() {
            return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        });
        if (e != cudaSuccess) return e;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((M + kTN - 1) / kTN, (N + kTM - 1) / kTM);
    cfg.blockDim = dim3(kTcThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = L.stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = L.pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kern, mw, mx, M, N, k0, steps, C, ldc, err);
}

}  // namespace

bool gemm_tc_supported(int K, int k_splits) { return K > 0 && K % (kTK * k_splits) == 0; }

cudaError_t launch_i8_to_f16(const int8_t* x, size_t n, uint16_t* y, const Launch& L) {
    if (n == 0) return cudaSuccess;
    if (n % 16 || (reinterpret_cast<uintptr_t>(x) & 15) || (reinterpret_cast<uintptr_t>(y) & 15))
        return cudaErrorInvalidValue;
    const size_t n16 = n / 16;
    const size_t blocks = std::min<size_t>((n16 + 255) / 256, (size_t)L.num_sms * 8);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)blocks);
    cfg.blockDim = dim3(256);
    cfg.stream = L.stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = L.pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, i8_to_f16_kernel, x, n16, y);
}

cudaError_t launch_gemm_tc(const uint16_t* X16, int M, const int8_t* W, int N, int K, int k0, int k1,
                           int32_t* C, int ldc, unsigned* err, const Launch& L) {
    if (M <= 0 || N <= 0 || k1 <= k0) return cudaSuccess;
    if ((k1 - k0) % kTK || k0 % kTK || K % 16 || (reinterpret_cast<uintptr_t>(X16) & 15) ||
        (reinterpret_cast<uintptr_t>(W) & 15))
        return cudaErrorInvalidValue;
    CUtensorMap mw, mx;
    if (!make_i8_map(&mw, W, N, K, K) || !make_f16_map(&mx, X16, M, K))
        return cudaErrorInvalidValue;
    return launch_tc_t<kStages8, kStages16>(mw, mx, M, N, k0, (k1 - k0) / kTK, C, ldc, err, L);
}

}  // namespace a8w8
