// Self-conditioning soft embedding E = gamma * P[:, s:e] W_shard[0:e-s], with
// P = bf16(exp(logits - lse)) formed on the fly in shared memory.
//
// What it computes: calvarado04.com, eq. e^sc (the expected embedding p_i W) and
// "The fix" (the product over a vocabulary slice [s, e) with the shard's first e-s
// rows, the probabilities cast to the embedding dtype, gamma applied after the sum;
// padded shard rows are never part of the product).
//
// Kernel design (one dense contraction on the 5th-generation tensor cores):
//   - a CTA owns an output tile of 128 rows x 256 columns and one contiguous range of
//     vocabulary blocks (split-K); the fp32 accumulator lives in tensor memory (256
//     TMEM columns);
//   - warp 0 streams, per 32-entry vocabulary block, the logits tile [128 x 32] fp32
//     and the W tile [32 x 256] bf16 into shared memory with TMA (128-byte swizzle);
//   - warps 2..5 turn the logits tile into the bf16 A operand, exp2(l*log2e - lse*log2e)
//     rounded to nearest even, written in the K-major 64-byte-swizzled layout the
//     tensor core reads; probabilities never go to global memory;
//   - warp 1 issues tcgen05.mma (M=128, N=256, K=16, bf16 x bf16 -> fp32), W being the
//     N-major B operand straight from the TMA tile; tcgen05.commit frees the stage;
//   - after the last block the same four warps read the accumulator back with
//     tcgen05.ld and store the partial tile; a second kernel adds the split partials
//     in split order, multiplies by gamma and writes E (deterministic).
//   Every barrier wait is bounded (about a second); a wait that gives up records
//   DG_ERR_TIMEOUT, drains what is in flight and leaves the kernel.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "dg_common.cuh"
#include "dg_internal.h"

namespace dg {

namespace {

constexpr int BM = 128;          // rows per tile (TMEM lanes)
constexpr int BN = 256;          // output columns per tile (one MMA N)
constexpr int BK = 32;           // vocabulary entries per stage
constexpr int STAGES = 5;
constexpr int THREADS = 192;     // warp 0: TMA, warp 1: MMA, warps 2..5: A producers + epilogue
constexpr int TMEM_COLS = 256;

constexpr int L_BYTES = BM * BK * 4;   // logits tile, rows of 128 B (128-byte swizzle)
constexpr int W_BOX_BYTES = BK * 64 * 2;
constexpr int W_BYTES = BK * BN * 2;   // 4 TMA boxes of [32 rows x 64 columns]
constexpr int A_BYTES = BM * BK * 2;   // bf16 probabilities, rows of 64 B (64-byte swizzle)
constexpr int STAGE_BYTES = L_BYTES + W_BYTES + A_BYTES;
constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + 1024 /*align*/ + 256 /*barriers*/;

static_assert(L_BYTES % 1024 == 0 && W_BYTES % 1024 == 0 && A_BYTES % 1024 == 0, "1 KiB alignment");

struct Params {
    const float *lse;
    float *ws;           // partial tiles
    int64_t k_begin;     // first vocabulary column of block 0 (multiple of 4)
    int64_t vocab_start;
    int64_t vocab_end;
    int64_t nkb;
    int R;
    int m_tiles, n_tiles, splits;
};

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

__global__ void __launch_bounds__(THREADS, 1)
    soft_embed_kernel(const __grid_constant__ CUtensorMap tm_logits, const __grid_constant__ CUtensorMap tm_w,
                      const Params p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + STAGES * STAGE_BYTES);
    uint64_t *full_tma = bars;               // TMA bytes landed (logits + W)
    uint64_t *full_a = bars + STAGES;        // A operand written by the 128 producer threads
    uint64_t *empty = bars + 2 * STAGES;     // MMA done with the stage
    uint64_t *acc_full = bars + 3 * STAGES;  // accumulator complete
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 3 * STAGES + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    const int bid = blockIdx.x;
    const int nt = bid % p.n_tiles;
    const int mt = (bid / p.n_tiles) % p.m_tiles;
    const int split = bid / (p.n_tiles * p.m_tiles);
    const int64_t kb0 = (int64_t)split * p.nkb / p.splits;
    const int64_t kb1 = (int64_t)(split + 1) * p.nkb / p.splits;
    const int nkb = (int)(kb1 - kb0);
    const int row0 = mt * BM;
    const int col0 = nt * BN;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(smem_u32(&full_tma[s]), 1);
            mbar_init(smem_u32(&full_a[s]), 128);
            mbar_init(smem_u32(&empty[s]), 1);
        }
        mbar_init(smem_u32(acc_full), 1);
        *abort_flag = 0;
        fence_mbar_init();
        prefetch_tmap(&tm_logits);
        prefetch_tmap(&tm_w);
    }
    __syncwarp();
    if (warp == 0) tmem_alloc<TMEM_COLS>(smem_u32(tmem_slot));
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            int issued[STAGES];
#pragma unroll
            for (int s = 0; s < STAGES; ++s) issued[s] = 0;
            bool ok = true;
            for (int i = 0; i < nkb; ++i) {
                const int s = i % STAGES;
                const uint32_t u = (uint32_t)(i / STAGES);
                if (u > 0 && !mbar_wait(smem_u32(&empty[s]), (u - 1) & 1, abort_flag)) {
                    ok = false;
                    break;
                }
                uint8_t *st = smem + s * STAGE_BYTES;
                const uint32_t bar = smem_u32(&full_tma[s]);
                mbar_arrive_expect_tx(bar, L_BYTES + W_BYTES);
                const int64_t k = p.k_begin + (kb0 + i) * BK;
                tma_load_2d(smem_u32(st), &tm_logits, bar, (int)k, row0);
                const int wy = (int)(k - p.vocab_start);
#pragma unroll
                for (int j = 0; j < BN / 64; ++j)
                    tma_load_2d(smem_u32(st + L_BYTES + j * W_BOX_BYTES), &tm_w, bar, col0 + 64 * j, wy);
                issued[s] = (int)u + 1;
            }
            if (!ok) {
                // let every copy already issued land before the CTA leaves
                for (int s = 0; s < STAGES; ++s)
                    if (issued[s] > 0) drain_wait(smem_u32(&full_tma[s]), (issued[s] - 1) & 1);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_bf16_f32(BM, BN, /*A K-major*/ 0, /*B N-major*/ 1);
            bool issued_any = false;
            for (int i = 0; i < nkb; ++i) {
                const int s = i % STAGES;
                const uint32_t ph = (uint32_t)(i / STAGES) & 1;
                if (!mbar_wait(smem_u32(&full_a[s]), ph, abort_flag)) break;
                if (!mbar_wait(smem_u32(&full_tma[s]), ph, abort_flag)) break;
                tc_fence_after();
                const uint32_t a_addr = smem_u32(smem + s * STAGE_BYTES + L_BYTES + W_BYTES);
                const uint32_t b_addr = smem_u32(smem + s * STAGE_BYTES + L_BYTES);
#pragma unroll
                for (int kk = 0; kk < BK / 16; ++kk) {
                    // A: K-major, 64-byte rows, 8-row groups 512 B apart; +32 B per K=16 step
                    const uint64_t a_desc = smem_desc(a_addr + kk * 32, 16, 512, 4);
                    // B: N-major, 64-column atoms 4 KiB apart (LBO), 8-row groups 1 KiB apart (SBO)
                    const uint64_t b_desc = smem_desc(b_addr + kk * 2048, W_BOX_BYTES, 1024, 2);
                    umma_bf16(tmem_base, a_desc, b_desc, idesc, (i > 0 || kk > 0) ? 1u : 0u);
                }
                umma_commit(smem_u32(&empty[s]));
                issued_any = true;
            }
            umma_commit(smem_u32(acc_full));
            if (*abort_flag && issued_any) drain_wait(smem_u32(acc_full), 0);
        }
    } else {
        // ------------------------------------------------------------ A producers, then epilogue
        const int quarter = warp & 3;  // TMEM lane quarter this warp may access
        const int r = quarter * 32 + lane;
        const int row = row0 + r;
        const bool valid_row = row < p.R;
        const float neg_lse2 = valid_row ? -p.lse[row] * kLog2e : 0.0f;
        bool ok = true;
        for (int i = 0; i < nkb; ++i) {
            const int s = i % STAGES;
            const uint32_t ph = (uint32_t)(i / STAGES) & 1;
            if (!mbar_wait(smem_u32(&full_tma[s]), ph, abort_flag)) {
                ok = false;
                break;
            }
            const uint8_t *lt = smem + s * STAGE_BYTES;
            uint8_t *at = smem + s * STAGE_BYTES + L_BYTES + W_BYTES;
            const int64_t k = p.k_begin + (kb0 + i) * BK;
            const bool edge = (k < p.vocab_start) || (k + BK > p.vocab_end);
            uint32_t packed[BK / 2];
#pragma unroll
            for (int c = 0; c < BK / 4; ++c) {
                const float4 v = *reinterpret_cast<const float4 *>(lt + r * 128 + ((c ^ (r & 7)) << 4));
                float e0 = ex2_approx(fmaf(v.x, kLog2e, neg_lse2));
                float e1 = ex2_approx(fmaf(v.y, kLog2e, neg_lse2));
                float e2 = ex2_approx(fmaf(v.z, kLog2e, neg_lse2));
                float e3 = ex2_approx(fmaf(v.w, kLog2e, neg_lse2));
                if (edge) {
                    const int64_t v0 = k + 4 * c;
                    if (v0 + 0 < p.vocab_start || v0 + 0 >= p.vocab_end) e0 = 0.f;
                    if (v0 + 1 < p.vocab_start || v0 + 1 >= p.vocab_end) e1 = 0.f;
                    if (v0 + 2 < p.vocab_start || v0 + 2 >= p.vocab_end) e2 = 0.f;
                    if (v0 + 3 < p.vocab_start || v0 + 3 >= p.vocab_end) e3 = 0.f;
                }
                if (!valid_row) e0 = e1 = e2 = e3 = 0.f;
                packed[2 * c] = pack_bf16x2(e0, e1);
                packed[2 * c + 1] = pack_bf16x2(e2, e3);
            }
#pragma unroll
            for (int c8 = 0; c8 < BK / 8; ++c8) {
                uint4 w = make_uint4(packed[4 * c8], packed[4 * c8 + 1], packed[4 * c8 + 2], packed[4 * c8 + 3]);
                *reinterpret_cast<uint4 *>(at + r * 64 + ((c8 ^ ((r >> 1) & 3)) << 4)) = w;
            }
            fence_proxy_async_smem();
            mbar_arrive(smem_u32(&full_a[s]));
        }
        // epilogue: accumulator -> partial tile, layout [BN/4 column groups][128 rows][4]
        float4 *dst = reinterpret_cast<float4 *>(p.ws) +
                      ((int64_t)(split * p.m_tiles + mt) * p.n_tiles + nt) * (BN / 4) * BM;
        // tcgen05.ld is warp-collective: the warp goes on only if every lane got here cleanly
        bool have_acc = false;
        if (nkb > 0 && __all_sync(0xffffffffu, ok)) {
            const bool got = mbar_wait(smem_u32(acc_full), 0, abort_flag);
            have_acc = __all_sync(0xffffffffu, got);
        }
        if (have_acc) {
            tc_fence_after();
            const uint32_t trow = tmem_base + ((uint32_t)(quarter * 32) << 16);
#pragma unroll 1
            for (int j = 0; j < BN / 32; ++j) {
                uint32_t v[32];
                tmem_ld_32x32b_x32(trow + j * 32, v);
                tmem_ld_wait();
#pragma unroll
                for (int c4 = 0; c4 < 8; ++c4) {
                    const float4 o = make_float4(__uint_as_float(v[4 * c4]), __uint_as_float(v[4 * c4 + 1]),
                                                 __uint_as_float(v[4 * c4 + 2]), __uint_as_float(v[4 * c4 + 3]));
                    dst[(j * 8 + c4) * BM + r] = o;
                }
            }
        } else if (nkb == 0) {
            for (int cg4 = 0; cg4 < BN / 4; ++cg4) dst[cg4 * BM + r] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc<TMEM_COLS>(tmem_base);
    }
}

// E[i, c] = gamma * sum over splits of the partial tiles, in split order.
__global__ void splitk_reduce_kernel(const float4 *__restrict__ ws, int splits, int m_tiles, int n_tiles, int R,
                                     int d, float gamma, float *__restrict__ out, int64_t ldo, int vec_out) {
    const int64_t groups = (int64_t)n_tiles * (BN / 4);  // column groups of 4
    const int64_t total = (int64_t)R * groups;
    const int64_t tile_stride = (int64_t)m_tiles * n_tiles * (BN / 4) * BM;
    for (int64_t t = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; t < total;
         t += (int64_t)gridDim.x * blockDim.x) {
        // consecutive threads take consecutive rows of one column group: coalesced reads
        const int64_t g = t / R;
        const int i = (int)(t - g * R);
        const int c = (int)(g * 4);
        if (c >= d) continue;
        const int mt = i / BM, r = i % BM;
        const int nt = (int)(g / (BN / 4)), cg = (int)(g % (BN / 4));
        const float4 *src = ws + ((int64_t)mt * n_tiles + nt) * (BN / 4) * BM + (int64_t)cg * BM + r;
        float4 acc = src[0];
        for (int s = 1; s < splits; ++s) {
            const float4 v = src[s * tile_stride];
            acc.x += v.x;
            acc.y += v.y;
            acc.z += v.z;
            acc.w += v.w;
        }
        float *o = out + (int64_t)i * ldo + c;
        if (vec_out && c + 4 <= d) {
            *reinterpret_cast<float4 *>(o) = make_float4(gamma * acc.x, gamma * acc.y, gamma * acc.z, gamma * acc.w);
        } else {
            const float a4[4] = {acc.x, acc.y, acc.z, acc.w};
            for (int e = 0; e < 4 && c + e < d; ++e) o[e] = gamma * a4[e];
        }
    }
}

PFN_cuTensorMapEncodeTiled_v12000 get_encode() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    });
    return fn;
}

}  // namespace

size_t soft_embed_workspace_bytes(const SoftEmbedPlan &plan, int splits) {
    return (size_t)splits * (size_t)plan.m_tiles * (size_t)plan.n_tiles * BM * BN * sizeof(float);
}

bool plan_soft_embed(int64_t R, int64_t vocab_start, int64_t vocab_end, int64_t d, int num_sms,
                     SoftEmbedPlan *plan) {
    if (R <= 0 || d <= 0 || vocab_end <= vocab_start || vocab_start < 0 || num_sms <= 0) return false;
    SoftEmbedPlan pl;
    pl.k_begin = vocab_start & ~int64_t(3);
    pl.nkb = (vocab_end - pl.k_begin + BK - 1) / BK;
    pl.m_tiles = (int)((R + BM - 1) / BM);
    pl.n_tiles = (int)((d + BN - 1) / BN);
    const int64_t tiles = (int64_t)pl.m_tiles * pl.n_tiles;
    int64_t splits = tiles >= num_sms ? 1 : num_sms / tiles;
    if (splits > pl.nkb) splits = pl.nkb;
    if (splits < 1) splits = 1;
    pl.splits = (int)splits;
    pl.workspace_bytes = soft_embed_workspace_bytes(pl, pl.splits);
    *plan = pl;
    return true;
}

cudaError_t launch_soft_embed(const float *logits, int64_t ldl, const float *lse, int64_t R, int64_t vocab_start,
                              int64_t vocab_end, const uint16_t *W, int64_t ldw, int64_t d, float gamma, float *out,
                              int64_t ldo, void *workspace, const SoftEmbedPlan &plan, cudaStream_t stream,
                              const char **msg) {
    PFN_cuTensorMapEncodeTiled_v12000 encode = get_encode();
    if (!encode) {
        *msg = "cuTensorMapEncodeTiled is not available from the driver";
        return cudaErrorNotSupported;
    }
    CUtensorMap tm_l, tm_w;
    {
        const cuuint64_t dims[2] = {(cuuint64_t)vocab_end, (cuuint64_t)R};
        const cuuint64_t strides[1] = {(cuuint64_t)ldl * 4};
        const cuuint32_t box[2] = {BK, BM};
        const cuuint32_t estr[2] = {1, 1};
        if (encode(&tm_l, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float *>(logits), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS) {
            *msg = "tensor map of the logits could not be encoded";
            return cudaErrorInvalidValue;
        }
    }
    {
        const cuuint64_t dims[2] = {(cuuint64_t)d, (cuuint64_t)(vocab_end - vocab_start)};
        const cuuint64_t strides[1] = {(cuuint64_t)ldw * 2};
        const cuuint32_t box[2] = {64, BK};
        const cuuint32_t estr[2] = {1, 1};
        if (encode(&tm_w, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t *>(W), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS) {
            *msg = "tensor map of the embedding shard could not be encoded";
            return cudaErrorInvalidValue;
        }
    }
    static std::once_flag attr_once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(attr_once, [] {
        attr_err = cudaFuncSetAttribute(soft_embed_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    });
    if (attr_err != cudaSuccess) {
        *msg = "could not raise the shared-memory limit of the soft-embed kernel";
        return attr_err;
    }
    Params p;
    p.lse = lse;
    p.ws = static_cast<float *>(workspace);
    p.k_begin = plan.k_begin;
    p.vocab_start = vocab_start;
    p.vocab_end = vocab_end;
    p.nkb = plan.nkb;
    p.R = (int)R;
    p.m_tiles = plan.m_tiles;
    p.n_tiles = plan.n_tiles;
    p.splits = plan.splits;
    const unsigned grid = (unsigned)(plan.splits * plan.m_tiles * plan.n_tiles);
    soft_embed_kernel<<<grid, THREADS, SMEM_BYTES, stream>>>(tm_l, tm_w, p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
        *msg = "soft-embed kernel launch failed";
        return e;
    }
    const int vec_out = (ldo % 4 == 0) && (((uintptr_t)out & 15) == 0);
    const int64_t total = R * (int64_t)plan.n_tiles * (BN / 4);
    int64_t blocks = (total + 255) / 256;
    const int64_t cap = (int64_t)device_sm_count() * 8;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    splitk_reduce_kernel<<<(unsigned)blocks, 256, 0, stream>>>(static_cast<const float4 *>(workspace), plan.splits,
                                                               plan.m_tiles, plan.n_tiles, (int)R, (int)d, gamma, out,
                                                               ldo, vec_out);
    e = cudaGetLastError();
    if (e != cudaSuccess) *msg = "split-K reduce launch failed";
    return e;
}

}  // namespace dg
