// gemv_mma.cu -- A8W8 decode projections for batches of 3 to 16 rows on the
// tensor cores, and the once-per-row activation quantisation they read.
//
// Same arithmetic as gemv.cu ("perf(qwen3-a8w8): optimize decode scheduling
// and data paths", pypto-lib PR #810, "Gate/Up INT8 path" and "Decode
// scheduling"): exact INT32 accumulators per K split, float32 dequantisation
// (acc * s_x) * s_w, residual or SwiGLU, one BF16 narrowing.
//
// Why tensor cores here: with a batch of 16 the dp4a GEMV reads every
// activation byte from shared memory once per batch row and weight byte and
// becomes ALU bound well below the HBM roofline. mma.sync m16n8k32 (INT8 x
// INT8 -> INT32, exact) multiplies the 16 batch rows (A) by 8 weight rows (B)
// per instruction, straight from the INT8 bytes. (tcgen05 has no INT8 kind
// on this architecture; an FP16 mma.sync on exact FP16 images of the codes
// measured the same time, so the INT8 form, which needs no conversion and no
// float chunking, is the one kept.)
//
// Layout and schedule (one CTA of 512 threads per SM):
//   * CTA c owns output channels [c*N/G, (c+1)*N/G) (both halves for
//     Gate/Up), cut into groups of 8 rows; groups are gathered into batches
//     of at most 8 (balanced), and K into steps of 64 columns.
//   * A slab is (group batch, K step). Each warp takes a contiguous run of
//     slabs. Per slab it loads the A fragment (16 batch rows x 64 columns of
//     INT8 codes, from L2) once and reuses it for up to 8 weight groups.
//   * Weight unit = 8 rows x 64 columns (512 bytes): lane (g, t) copies the
//     16 bytes of row g at column 16 t into a private shared-memory ring with
//     cp.async, 16 units ahead (one commit group per unit); its four words
//     are the B fragments of two m16n8k32 instructions. The K columns are
//     permuted inside a step (the same permutation for A), which a sum does
//     not see. Each warp's INT32 tiles are added into the CTA's accumulators
//     in shared memory (atomics, exact) at batch and split boundaries.
//   * The activation rows are quantised once, by quant_prep_kernel (one CTA
//     per row, RMSNorm optional, the same code as the dp4a prologue), not
//     once per CTA.
#include "gemv_impl.cuh"

namespace a8w8 {

namespace {

using namespace gemv;

constexpr int kMmaThreads = 512;
constexpr int kMmaRows = 16;      // batch rows per launch (the MMA's M)
constexpr int kMmaStep = 64;      // K columns per step
constexpr int kMmaGroupsMax = 8;  // weight groups per batch
constexpr int kMmaNB = 16;        // ring depth, units per lane (16 copies in flight)
constexpr int kMmaNBPre = 8;      // units requested before the dependency wait
constexpr size_t kMmaRingBytes = (size_t)kMmaNB * kMmaThreads * 16;
constexpr int kMaxDynSmem = 227 * 1024;
constexpr int kPrepThreads = 1024;  // one CTA per row, the batch-1 prologue's width

__device__ __forceinline__ void mma_s8_16832(int (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                             uint32_t a3, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k32.row.col.s32.s8.s8.s32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
        "{%8, %9}, {%0, %1, %2, %3};"
        : "+r"(d[0]), "+r"(d[1]), "+r"(d[2]), "+r"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void cp_async16_zf(uint32_t s, const void* g, int src_bytes,
                                              uint64_t policy) {
    asm volatile("cp.async.cg.shared.global.L2::cache_hint [%0], [%1], 16, %2, %3;" ::"r"(s), "l"(g),
                 "r"(src_bytes), "l"(policy)
                 : "memory");
}

struct MmaSmem {
    size_t accs, xs, ring, total;
};
__host__ __device__ inline MmaSmem mma_smem(int nseg, int KS, int N, int G) {
    const int rows_max = (N + G - 1) / G;
    MmaSmem s;
    s.accs = 0;
    s.xs = align16((size_t)nseg * rows_max * KS * kMmaRows * 4);
    s.ring = (s.xs + kMmaRows * 4 + 127) & ~size_t(127);
    s.total = s.ring + kMmaRingBytes;
    return s;
}

template <int EPI, int KS>
__global__ void __launch_bounds__(kMmaThreads, 1) gemv_mma_kernel(const GemvParams p) {
    extern __shared__ __align__(16) unsigned char smem[];
    constexpr int NSEG = (EPI == EPI_SWIGLU) ? 2 : 1;
    constexpr int NW = kMmaThreads / 32;
    constexpr int GM = kMmaGroupsMax;
    const int K = p.K, N = p.N, M = p.M;
    const int G = gridDim.x;
    const int o0 = (int)(((long long)N * blockIdx.x) / G);
    const int o1 = (int)(((long long)N * (blockIdx.x + 1)) / G);
    const int nrows = o1 - o0;
    const int rows_max = (N + G - 1) / G;
    const MmaSmem L = mma_smem(NSEG, KS, N, G);
    int32_t* accs = reinterpret_cast<int32_t*>(smem + L.accs);
    float* xs = reinterpret_cast<float*>(smem + L.xs);
    const uint32_t ring = (uint32_t)__cvta_generic_to_shared(smem + L.ring) + threadIdx.x * 16u;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, t = lane & 3;
    const int G8 = (nrows + 7) / 8;              // groups per segment
    const int TG = NSEG * G8;                    // groups
    const int NBAT = (TG + GM - 1) / GM;         // batches of <= 8 groups
    const int KST = K / kMmaStep;                // steps per row
    const int kps = KST / KS;                    // steps per split
    const int S = NBAT * KST;                    // slabs (batch, step)
    const int s0 = (int)(((long long)S * warp) / NW);
    const int s1 = (int)(((long long)S * (warp + 1)) / NW);

    // Issue cursor, one weight unit per call: slab i_sl = (batch i_bt, step
    // i_st), group i_gg of [i_ga, i_ge); divisions only when the batch changes.
    int i_sl = s0, i_bt = 0, i_st = 0, i_ga = 0, i_ge = 0, i_gg = 0;
    if (s0 < s1) {
        i_bt = s0 / KST;
        i_st = s0 - i_bt * KST;
        i_ga = i_bt * TG / NBAT;
        i_ge = (i_bt + 1) * TG / NBAT;
        i_gg = i_ga;
    }
    const uint64_t pol = l2_evict_first_policy();
    int wslot = 0;
    auto issue = [&]() {
        if (i_sl < s1) {
            const int seg = (NSEG == 2 && i_gg >= G8) ? 1 : 0;
            const int r = 8 * (i_gg - seg * G8) + g;
            const bool ok = r < nrows;
            const int8_t* src = p.W + (size_t)(seg * N + o0 + (ok ? r : 0)) * K +
                                (size_t)i_st * kMmaStep + 16 * t;
            cp_async16_zf(ring + (uint32_t)(wslot * kMmaThreads * 16), src, ok ? 16 : 0, pol);
            if (++i_gg == i_ge) {
                ++i_sl;
                if (++i_st == KST) {
                    i_st = 0;
                    ++i_bt;
                    i_ga = i_bt * TG / NBAT;
                    i_ge = (i_bt + 1) * TG / NBAT;
                }
                i_gg = i_ga;
            }
        }
        cp_async_commit();
        wslot = wslot + 1 == kMmaNB ? 0 : wslot + 1;
    };
#pragma unroll 1
    for (int i = 0; i < kMmaNBPre; ++i) issue();

    pdl_wait();
    pdl_trigger();

    if (p.clear && blockIdx.x == 0)
        for (int i = threadIdx.x; i < p.clear_n; i += kMmaThreads) p.clear[i] = 0u;
    const int acc_n = NSEG * rows_max * KS * kMmaRows;
    for (int i = threadIdx.x; i < acc_n; i += kMmaThreads) accs[i] = 0;
    if (threadIdx.x < kMmaRows)
        xs[threadIdx.x] = (int)threadIdx.x < M ? __ldcg(p.x_scale + threadIdx.x) : 0.0f;
#pragma unroll 1
    for (int i = kMmaNBPre; i < kMmaNB; ++i) issue();
    __syncthreads();

    // A rows g and g + 8 of a step (16 bytes each; zero beyond M)
    const int8_t* xa = p.xq + (size_t)g * K + 16 * t;
    const int8_t* xb = p.xq + (size_t)(g + 8) * K + 16 * t;
    const bool ra = g < M, rb = g + 8 < M;
    auto load_a = [&](int step, int4& a, int4& b) {
        a = ra ? ld_cg_v4(xa + (size_t)step * kMmaStep) : make_int4(0, 0, 0, 0);
        b = rb ? ld_cg_v4(xb + (size_t)step * kMmaStep) : make_int4(0, 0, 0, 0);
    };

    int c[GM][4];
#pragma unroll
    for (int j = 0; j < GM; ++j) c[j][0] = c[j][1] = c[j][2] = c[j][3] = 0;

    // consumer cursor: batch bt (groups [ga, ga + ng)), step st
    int bt = 0, st = 0, ga = 0, ng = 0;
    if (s0 < s1) {
        bt = s0 / KST;
        st = s0 - bt * KST;
        ga = bt * TG / NBAT;
        ng = (bt + 1) * TG / NBAT - ga;
    }
    int rslot = 0;
    int4 na = make_int4(0, 0, 0, 0), nb = na;
    if (s0 < s1) load_a(st, na, nb);
    int split = KS == 1 ? 0 : st / kps;
#pragma unroll 1
    for (int sl = s0; sl < s1; ++sl) {
        // A fragments of this step (rows g and g + 8), the next step's loads
        // in flight. MMA m of the step: logical columns 4t..4t+3 <- the
        // lane's word 2m, 16+4t..16+4t+3 <- word 2m + 1 (A and B alike).
        const uint32_t wa[4] = {(uint32_t)na.x, (uint32_t)na.y, (uint32_t)na.z, (uint32_t)na.w};
        const uint32_t wb[4] = {(uint32_t)nb.x, (uint32_t)nb.y, (uint32_t)nb.z, (uint32_t)nb.w};
        const int nst = st + 1 == KST ? 0 : st + 1;
        if (sl + 1 < s1) load_a(nst, na, nb);
#pragma unroll
        for (int j = 0; j < GM; ++j) {
            if (j < ng) {
                cp_async_wait_group<kMmaNB - 1>();
                const int4 w = lds_v4(ring + (uint32_t)(rslot * kMmaThreads * 16));
                rslot = rslot + 1 == kMmaNB ? 0 : rslot + 1;
                issue();   // refill the slot just read
                mma_s8_16832(c[j], wa[0], wb[0], wa[1], wb[1], (uint32_t)w.x, (uint32_t)w.y);
                mma_s8_16832(c[j], wa[2], wb[2], wa[3], wb[3], (uint32_t)w.z, (uint32_t)w.w);
            }
        }
        const bool last = sl + 1 == s1;
        const bool batch_end = nst == 0;
        const bool split_end = KS == 2 && st + 1 == kps;
        if (last || batch_end || split_end) {
            // INT32 tiles -> shared accumulators
#pragma unroll
            for (int j = 0; j < GM; ++j) {
                if (j < ng) {
                    const int gg = ga + j;
                    const int seg = (NSEG == 2 && gg >= G8) ? 1 : 0;
                    const int r0 = 8 * (gg - seg * G8) + 2 * t;
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int r = r0 + (e & 1);
                        const int b = g + ((e >> 1) << 3);
                        if (r < nrows && b < M)
                            atomicAdd(&accs[((seg * rows_max + r) * KS + split) * kMmaRows + b], c[j][e]);
                        c[j][e] = 0;
                    }
                }
            }
        }
        if (split_end) split = 1;
        if (batch_end) {
            ++bt;
            ga = bt * TG / NBAT;
            ng = (bt + 1) * TG / NBAT - ga;
            split = 0;
        }
        st = nst;
    }
    cp_async_wait_all();
    __syncthreads();
    epilogue<kMmaRows, EPI, KS>(p, accs, xs, o0, nrows, rows_max, nullptr, false);
}

// One CTA per activation row: the dp4a prologue's quantisation (RMSNorm
// optional) for that row, written to global memory for the MMA projections.
template <int PRO>
__global__ void __launch_bounds__(kPrepThreads) quant_prep_kernel(const GemvParams p, int8_t* xq,
                                                                  float* xsc) {
    extern __shared__ __align__(16) unsigned char smem[];
    const int b = blockIdx.x, K = p.K;
    const SmemLayout L = smem_layout(1, 1, 1, K, 1, 1, kPrepThreads);
    int8_t* act = reinterpret_cast<int8_t*>(smem + L.act);
    float* xs = reinterpret_cast<float*>(smem + L.xs);
    float* red = reinterpret_cast<float*>(smem + L.red);
    bf16* stage = L.stage ? reinterpret_cast<bf16*>(smem + L.stage) : nullptr;
    GemvParams q = p;
    q.M = 1;
    q.x = p.x + (size_t)b * p.ldx;
    q.tap_x = nullptr;
    q.tap_q = nullptr;
    q.tap_s = nullptr;
    pdl_wait();
    pdl_trigger();
    int4 nwr[1];
    prologue<1, PRO, 1>(q, act, xs, red, stage, nwr, false, [] {});
    const int vec = K / 16;
    for (int j = threadIdx.x; j < vec; j += kPrepThreads) {
        const int4 v = *reinterpret_cast<const int4*>(act + 16 * j);
        *reinterpret_cast<int4*>(xq + (size_t)b * K + 16 * j) = v;
        if (p.tap_q) *reinterpret_cast<int4*>(p.tap_q + (size_t)b * K + 16 * j) = v;
    }
    if (PRO == PRO_NORM_QUANT && p.tap_x && stage) {
        for (int j = threadIdx.x; j < K / 8; j += kPrepThreads)
            *reinterpret_cast<int4*>(p.tap_x + (size_t)b * K + 8 * j) =
                *reinterpret_cast<const int4*>(stage + 8 * j);
    }
    if (threadIdx.x == 0) {
        xsc[b] = xs[0];
        if (p.tap_s) p.tap_s[b] = xs[0];
    }
}

template <typename Kern>
cudaError_t launch_k(Kern kern, int grid, int block, size_t smem, const GemvParams& p,
                     const Launch& L) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(block);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = L.stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = L.pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kern, p);
}

template <int EPI, int KS>
cudaError_t launch_mma_t(const GemvParams& p, const Launch& L) {
    const int G = L.num_sms;
    const size_t smem = mma_smem(EPI == EPI_SWIGLU ? 2 : 1, KS, p.N, G).total;
    if (smem > (size_t)kMaxDynSmem) return cudaErrorInvalidValue;
    {
        // the shared-memory limit, set once per CUDA context
        cudaError_t e = once_per_context(reinterpret_cast<const void*>(gemv_mma_kernel<EPI, KS>), [&]() -> cudaError_t {
            cudaError_t e = cudaFuncSetAttribute(gemv_mma_kernel<EPI, KS>,
                                                 cudaFuncAttributeMaxDynamicSharedMemorySize, kMaxDynSmem);
            return e;
        });
        if (e != cudaSuccess) return e;
    }
    return launch_k(gemv_mma_kernel<EPI, KS>, G, kMmaThreads, smem, p, L);
}

template <int PRO>
cudaError_t launch_prep_t(const GemvParams& p, int8_t* xq, float* xs, const Launch& L) {
    const size_t smem = smem_layout(1, 1, 1, p.K, 1, 1, kPrepThreads).total;
    if (smem > (size_t)kMaxDynSmem) return cudaErrorInvalidValue;
    {
        // the shared-memory limit, set once per CUDA context
        cudaError_t e = once_per_context(reinterpret_cast<const void*>(quant_prep_kernel<PRO>), [&]() -> cudaError_t {
            cudaError_t e = cudaFuncSetAttribute(quant_prep_kernel<PRO>,
                                                 cudaFuncAttributeMaxDynamicSharedMemorySize, kMaxDynSmem);
            return e;
        });
        if (e != cudaSuccess) return e;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.M);
    cfg.blockDim = dim3(kPrepThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = L.stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = L.pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, quant_prep_kernel<PRO>, p, xq, xs);
}

}  // namespace

bool gemv_mma_supported(int K, int k_splits) {
    return K > 0 && K % (kMmaStep * k_splits) == 0;
}

cudaError_t launch_gemv_mma(int epilogue, int k_splits, const GemvParams& p, const Launch& L) {
    if (p.M <= 0) return cudaSuccess;
    if (p.M > kMmaRows || !p.xq || !p.x_scale || !gemv_mma_supported(p.K, k_splits))
        return cudaErrorInvalidValue;
    if (epilogue == EPI_STORE) {
        if (k_splits == 1) return launch_mma_t<EPI_STORE, 1>(p, L);
        if (k_splits == 2) return launch_mma_t<EPI_STORE, 2>(p, L);
        return cudaErrorInvalidValue;
    }
    if (k_splits != 1) return cudaErrorInvalidValue;
    return launch_mma_t<EPI_SWIGLU, 1>(p, L);
}

cudaError_t launch_quant_prep(int prologue, const GemvParams& p, int8_t* xq, float* xs,
                              const Launch& L) {
    if (p.M <= 0) return cudaSuccess;
    if (p.K % 16) return cudaErrorInvalidValue;
    if (prologue == PRO_NORM_QUANT) return launch_prep_t<PRO_NORM_QUANT>(p, xq, xs, L);
    if (prologue == PRO_QUANT) return launch_prep_t<PRO_QUANT>(p, xq, xs, L);
    return cudaErrorInvalidValue;
}

}  // namespace a8w8
