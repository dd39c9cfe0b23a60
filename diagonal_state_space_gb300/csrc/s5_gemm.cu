// s5_gemm.cu -- the dense bf16 contractions of the layer stack on the
// 5th-generation tensor cores: C[M][N] (fp32, row-major) = op(A) op(B) with
// bf16 operands and fp32 accumulation (the wiki summary's "Method" step 4 and
// gated pseudocode; the review's rows 1 and 4: B_bar z, the readout over X, the
// gate's W h, and their adjoints).
//
// Operands are row-major in global memory.  A is [M][K] (K-major) or, with
// ta, [K][M] (MN-major); B is [K][N] (MN-major) or, with tb, [N][K]
// (K-major).  Both layouts are read by TMA into the 128-byte-swizzle shared
// layout the MMA descriptors describe:
//   K-major   rows = M (or N), 128 B = 64 K-elements per row; 8-row groups
//             1024 B apart; a K-step of 16 advances the start by 32 B
//   MN-major  rows = K, 128 B = 64 M- (or N-) elements per row, in chunks of
//             64 K-rows (8 KB); 8-row groups 1024 B apart, chunks of 64
//             M-elements 8 KB apart; a K-step of 16 advances the start by 2 KB
//
// Kernel: persistent, one CTA per SM, tiles of 128 x 256 (one M=128, N=256,
// K=16 MMA per K-step), 64-deep K-blocks through a 4-stage ring.
//   warp 0      TMA producer (one elected thread)
//   warp 1      TMEM allocation and MMA issue (one elected thread); two
//               accumulators of 256 columns, so that the epilogue of a tile
//               overlaps the MMAs of the next
//   warps 2-5   epilogue: thread = accumulator row = TMEM lane; 32 columns
//               per load, written into a 128-byte-swizzled 32 x 32 block in
//               shared memory and sent out by one TMA store per block (two
//               blocks per warp in flight); rows and columns past M, N are
//               clipped by the copy
// When the output tiles alone cannot fill the SMs and K is long (the weight
// gradients, K = B*L), K is split over CTAs and the blocks are added into a
// zeroed C with TMA reduce-add copies.
// Every wait is bounded: a wait that runs out sets a device flag, and the
// kernel finishes without waiting further (the host reports the error).
// Shapes whose leading dimensions TMA cannot address (row pitch not a
// multiple of 16 bytes, unaligned bases) run on a plain CUDA-core kernel.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <cstring>
#include <mutex>

#include "s5_internal.cuh"
#include "s5_sm100.cuh"

namespace s5 {
using namespace sm100;

namespace {

constexpr int BM = 128, BN = 256, BK = 64;
constexpr int GSTAGES = 4;
constexpr int GTHREADS = 192;
constexpr uint32_t A_BYTES = BM * BK * 2;   // 16 KB
constexpr uint32_t B_BYTES = BN * BK * 2;   // 32 KB
constexpr uint32_t STAGE_BYTES = A_BYTES + B_BYTES;
// epilogue staging: per epilogue warp two buffers of 32 rows x 32 fp32 (4 KB)
constexpr uint32_t G_SM_OUT = GSTAGES * STAGE_BYTES;
constexpr uint32_t OUT_BUF = 32 * 32 * 4;
constexpr uint32_t G_SM_BAR = G_SM_OUT + 4 * 2 * OUT_BUF;
constexpr uint32_t G_SMEM = G_SM_BAR + 256 + 1024;   // + barriers + alignment slack
constexpr unsigned long long G_WAIT_NS = 2000000000ull;

__device__ int g_gemm_fault = 0;   // a bounded wait ran out

struct GemmBars {
    uint64_t full[GSTAGES], empty[GSTAGES];
    uint64_t acc_full[2], acc_empty[2];
    uint64_t drain;   // every MMA issued has completed (before TMEM is freed)
    uint32_t tmem_base;
    int abort;
};

// Shared-memory descriptor of a 128-byte-swizzle operand: start address,
// leading-dimension offset (MN-major: the stride of 64-element chunks along
// M or N), stride offset (8-row groups).
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr >> 4) & 0x3FFFu);
    d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
    d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
    d |= (uint64_t)1u << 46;
    d |= (uint64_t)2u << 61;
    return d;
}

__device__ __forceinline__ bool gemm_wait(uint64_t *bar, uint32_t parity, GemmBars *gb) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = global_ns();
    for (;;) {
        if (mbar_try_wait_sleep(bar, parity, 1000000)) return true;
        if (*reinterpret_cast<volatile int *>(&gb->abort)) return false;
        if (global_ns() - t0 > G_WAIT_NS) {
            *reinterpret_cast<volatile int *>(&gb->abort) = 1;
            atomicExch(&g_gemm_fault, 1);
            return false;
        }
    }
}

__device__ __forceinline__ void tma_load_2d(void *dst, const void *tmap, int c0, int c1, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_addr(dst)),
        "l"(reinterpret_cast<uint64_t>(tmap)), "r"(c0), "r"(c1), "r"(smem_addr(bar))
        : "memory");
}

__device__ __forceinline__ void tma_store_2d(const void *tmap, const void *src, int c0, int c1) {
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.tile.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
                     reinterpret_cast<uint64_t>(tmap)),
                 "r"(c0), "r"(c1), "r"(smem_addr(src))
                 : "memory");
}
__device__ __forceinline__ void tma_reduce_add_2d(const void *tmap, const void *src, int c0, int c1) {
    asm volatile("cp.reduce.async.bulk.tensor.2d.global.shared::cta.add.tile.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
                     reinterpret_cast<uint64_t>(tmap)),
                 "r"(c0), "r"(c1), "r"(smem_addr(src))
                 : "memory");
}
// Waits until at most one committed bulk group is still reading shared memory.
__device__ __forceinline__ void bulk_wait_read_1() {
    asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
}
__device__ __forceinline__ void sts128(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

struct GemmArgs {
    float *C;
    long long ldc;
    int M, N, K;
    int tiles_m, tiles_n, splits, kb_per_split;
    bool ta, tb, vec_ok;   // vec_ok: C rows 16-byte aligned (ldc % 4 == 0, C aligned)
};

__global__ void __launch_bounds__(GTHREADS, 1)
gemm_tc_kernel(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_b,
               const __grid_constant__ CUtensorMap tmap_c, const GemmArgs g) {
    extern __shared__ __align__(1024) unsigned char gsm_raw[];
    const uint32_t pad = (1024u - (smem_addr(gsm_raw) & 1023u)) & 1023u;
    unsigned char *smem = gsm_raw + pad;
    GemmBars *gb = reinterpret_cast<GemmBars *>(smem + G_SM_BAR);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int ntiles = g.tiles_m * g.tiles_n * g.splits;
    const int nkb_total = (g.K + BK - 1) / BK;

    if (threadIdx.x == 0) {
        for (int s = 0; s < GSTAGES; ++s) {
            mbar_init(&gb->full[s], 1);
            mbar_init(&gb->empty[s], 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(&gb->acc_full[a], 1);
            mbar_init(&gb->acc_empty[a], 4);
        }
        mbar_init(&gb->drain, 1);
        gb->abort = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(&gb->tmem_base, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = gb->tmem_base;

    // tile t: n fastest (the A row block is read by consecutive tiles), then
    // m, then the K split
    auto coords = [&](int t, int &m0, int &n0, int &kb0, int &kb1) {
        const int tn = t % g.tiles_n, r = t / g.tiles_n;
        const int tm = r % g.tiles_m, sp = r / g.tiles_m;
        m0 = tm * BM;
        n0 = tn * BN;
        kb0 = sp * g.kb_per_split;
        kb1 = min(nkb_total, kb0 + g.kb_per_split);
    };

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        int it = 0;   // k-blocks issued so far (ring position)
        bool ok = true;
        for (int t = blockIdx.x; ok && t < ntiles; t += gridDim.x) {
            int m0, n0, kb0, kb1;
            coords(t, m0, n0, kb0, kb1);
            for (int kb = kb0; kb < kb1; ++kb, ++it) {
                const int s = it % GSTAGES;
                if (it >= GSTAGES) {
                    ok = __shfl_sync(0xffffffffu, (int)gemm_wait(&gb->empty[s], ((it / GSTAGES) - 1) & 1, gb), 0);
                    if (!ok) break;
                }
                if (elect_one()) {
                    unsigned char *sa = smem + s * STAGE_BYTES, *sbp = sa + A_BYTES;
                    mbar_arrive_tx(&gb->full[s], STAGE_BYTES);
                    const int k0 = kb * BK;
                    if (!g.ta) {
                        tma_load_2d(sa, &tmap_a, k0, m0, &gb->full[s]);
                    } else {
                        tma_load_2d(sa, &tmap_a, m0, k0, &gb->full[s]);
                        tma_load_2d(sa + 8192, &tmap_a, m0 + 64, k0, &gb->full[s]);
                    }
                    if (g.tb) {
                        tma_load_2d(sbp, &tmap_b, k0, n0, &gb->full[s]);
                    } else {
#pragma unroll
                        for (int c = 0; c < 4; ++c) tma_load_2d(sbp + 8192 * c, &tmap_b, n0 + 64 * c, k0, &gb->full[s]);
                    }
                }
                __syncwarp();
            }
        }
        // copies in flight must land before the CTA exits
        for (int j = max(0, it - GSTAGES); j < it; ++j) {
            const unsigned long long t0 = global_ns();
            while (!mbar_try_wait_sleep(&gb->full[j % GSTAGES], (j / GSTAGES) & 1, 1000000))
                if (global_ns() - t0 > 200000000ull) break;
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issue
        const uint32_t idesc = idesc_bf16_f32(BM, BN) | ((g.ta ? 1u : 0u) << 15) | ((g.tb ? 0u : 1u) << 16);
        int it = 0, lt = 0;
        bool ok = true;
        for (int t = blockIdx.x; ok && t < ntiles; t += gridDim.x, ++lt) {
            int m0, n0, kb0, kb1;
            coords(t, m0, n0, kb0, kb1);
            const int ab = lt & 1;
            if (lt >= 2) {
                ok = __shfl_sync(0xffffffffu, (int)gemm_wait(&gb->acc_empty[ab], ((lt >> 1) - 1) & 1, gb), 0);
                if (!ok) break;
            }
            tc_fence_after();
            const uint32_t d = tmem + (uint32_t)ab * 256u;
            for (int kb = kb0; kb < kb1; ++kb, ++it) {
                const int s = it % GSTAGES;
                ok = __shfl_sync(0xffffffffu, (int)gemm_wait(&gb->full[s], (it / GSTAGES) & 1, gb), 0);
                if (!ok) break;
                tc_fence_after();
                const uint32_t sa = smem_addr(smem + s * STAGE_BYTES), sbp = sa + A_BYTES;
                if (elect_one()) {
#pragma unroll
                    for (int kk = 0; kk < BK / 16; ++kk) {
                        const uint64_t da = g.ta ? sw128_desc(sa + 2048u * kk, 8192u, 1024u)
                                                 : sw128_desc(sa + 32u * kk, 16u, 1024u);
                        const uint64_t db = g.tb ? sw128_desc(sbp + 32u * kk, 16u, 1024u)
                                                 : sw128_desc(sbp + 2048u * kk, 8192u, 1024u);
                        mma_bf16(d, da, db, idesc, (kb > kb0 || kk > 0) ? 1u : 0u);
                    }
                    mma_commit(&gb->empty[s]);
                }
                __syncwarp();
            }
            if (!ok) break;
            if (elect_one()) mma_commit(&gb->acc_full[ab]);
            __syncwarp();
        }
        // every MMA issued must complete before TMEM is freed (after a wait
        // gave up, some may still be in flight): bounded wait on a last commit
        if (elect_one()) mma_commit(&gb->drain);
        __syncwarp();
        const unsigned long long t0 = global_ns();
        while (!mbar_try_wait_sleep(&gb->drain, 0, 1000000))
            if (global_ns() - t0 > 200000000ull) break;
    } else {
        // ------------------------------------------------------------ epilogue
        const int q = warp & 3;   // TMEM lane quarter of this warp
        const uint32_t lane_base = tmem + ((uint32_t)(32 * q) << 16);
        const uint32_t out0 = smem_addr(smem + G_SM_OUT + (uint32_t)(q * 2) * OUT_BUF);
        int nblk = 0;   // output blocks this warp has staged
        int lt = 0;
        for (int t = blockIdx.x; t < ntiles; t += gridDim.x, ++lt) {
            int m0, n0, kb0, kb1;
            coords(t, m0, n0, kb0, kb1);
            const int ab = lt & 1;
            const bool ok = __all_sync(0xffffffffu, gemm_wait(&gb->acc_full[ab], (lt >> 1) & 1, gb));
            if (!ok) break;
            tc_fence_after();
            if (g.vec_ok) {
                // 32 x 32 blocks through shared memory: this thread's row r of
                // the block, 16-byte chunk j at (j ^ (r & 7)) (the copy's
                // 128-byte swizzle)
#pragma unroll 1
                for (int c0 = 0; c0 < BN; c0 += 32, ++nblk) {
                    uint32_t v[32];
                    tmem_ld32(lane_base + (uint32_t)ab * 256u + (uint32_t)c0, v);
                    const int buf = nblk & 1;
                    // the copy that last read this buffer (two blocks ago) must be done with it
                    if (elect_one()) bulk_wait_read_1();
                    __syncwarp();
                    tmem_wait_ld();
                    const uint32_t base = out0 + (uint32_t)buf * OUT_BUF + (uint32_t)lane * 128u;
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        sts128(base + (uint32_t)((j ^ (lane & 7)) << 4), v[4 * j], v[4 * j + 1], v[4 * j + 2],
                               v[4 * j + 3]);
                    fence_proxy_async_smem();
                    __syncwarp();
                    // one committed group per block (empty when the block lies
                    // wholly past N or M), so that "all but the last group"
                    // always covers the block two back
                    if (elect_one()) {
                        if (n0 + c0 < g.N && m0 + 32 * q < g.M) {
                            unsigned char *src = smem + G_SM_OUT + (uint32_t)(q * 2 + buf) * OUT_BUF;
                            if (g.splits > 1)
                                tma_reduce_add_2d(&tmap_c, src, n0 + c0, m0 + 32 * q);
                            else
                                tma_store_2d(&tmap_c, src, n0 + c0, m0 + 32 * q);
                        }
                        bulk_commit();
                    }
                    __syncwarp();
                }
            } else {
                const int row = m0 + 32 * q + lane;
                float *crow = g.C + (long long)row * g.ldc;
#pragma unroll 1
                for (int c0 = 0; c0 < BN; c0 += 32) {
                    uint32_t v[32];
                    tmem_ld32(lane_base + (uint32_t)ab * 256u + (uint32_t)c0, v);
                    tmem_wait_ld();
                    const int col = n0 + c0;
                    if (row < g.M && col < g.N) {
#pragma unroll
                        for (int j = 0; j < 32; ++j) {
                            if (col + j < g.N) {
                                if (g.splits > 1)
                                    atomicAdd(crow + col + j, __uint_as_float(v[j]));
                                else
                                    crow[col + j] = __uint_as_float(v[j]);
                            }
                        }
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&gb->acc_empty[ab]);
        }
        // the output copies must be complete before the kernel ends
        if (elect_one()) bulk_wait_all();
        __syncwarp();
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, 512);   // the MMA warp drained its MMAs above
}

// Plain CUDA-core GEMM for shapes TMA cannot address: 32 x 32 output tiles,
// 32-deep K slabs staged in shared memory.
__global__ void gemm_simt_kernel(const __nv_bfloat16 *__restrict__ A, long long lda,
                                 const __nv_bfloat16 *__restrict__ B, long long ldb, float *__restrict__ C,
                                 long long ldc, int M, int N, int K, bool ta, bool tb) {
    __shared__ float as[32][33], bs[32][33];
    const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;   // 32 x 8 threads
    const int m0 = blockIdx.y * 32, n0 = blockIdx.x * 32;
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    for (int k0 = 0; k0 < K; k0 += 32) {
        for (int r = ty; r < 32; r += 8) {
            // as[r][tx] = op(A)[m0 + r][k0 + tx], bs[r][tx] = op(B)[k0 + r][n0 + tx]
            const int m = m0 + r, k = k0 + tx;
            float av = 0.f;
            if (m < M && k < K) av = __bfloat162float(ta ? A[(long long)k * lda + m] : A[(long long)m * lda + k]);
            as[r][tx] = av;
            const int kk = k0 + r, n = n0 + tx;
            float bv = 0.f;
            if (kk < K && n < N) bv = __bfloat162float(tb ? B[(long long)n * ldb + kk] : B[(long long)kk * ldb + n]);
            bs[r][tx] = bv;
        }
        __syncthreads();
#pragma unroll 8
        for (int k = 0; k < 32; ++k) {
            const float b = bs[k][tx];
#pragma unroll
            for (int i = 0; i < 4; ++i) acc[i] = fmaf(as[ty + 8 * i][k], b, acc[i]);
        }
        __syncthreads();
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int m = m0 + ty + 8 * i, n = n0 + tx;
        if (m < M && n < N) C[(long long)m * ldc + n] = acc[i];
    }
}

PFN_cuTensorMapEncodeTiled_v12000 gemm_encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    return fn;
}

// Encoded tensor maps are cached by what they encode: the stack calls the
// same products on the same buffers every step, and encoding is host work.
struct MapKey {
    const void *base;
    long long rows, cols, ld;
    int box_rows, dtype;
    bool operator==(const MapKey &o) const {
        return base == o.base && rows == o.rows && cols == o.cols && ld == o.ld && box_rows == o.box_rows &&
               dtype == o.dtype;
    }
};
constexpr int MAP_CACHE = 256;
std::mutex g_map_mu;
MapKey g_map_keys[MAP_CACHE];
CUtensorMap g_map_vals[MAP_CACHE];
int g_map_used = 0, g_map_next = 0;

// 2-D map of a row-major [rows][cols] matrix with row pitch ld elements; box
// {box_cols columns, box_rows rows}, 128-byte swizzle, zero fill.  dtype 0:
// bf16 (box_cols 64), 1: fp32 (box_cols 32).
bool cached_map(CUtensorMap *map, const void *base, long long rows, long long cols, long long ld, int box_rows,
                int dtype) {
    const MapKey key{base, rows, cols, ld, box_rows, dtype};
    std::lock_guard<std::mutex> lk(g_map_mu);
    for (int i = 0; i < g_map_used; ++i)
        if (g_map_keys[i] == key) {
            *map = g_map_vals[i];
            return true;
        }
    auto fn = gemm_encode_fn();
    if (!fn) return false;
    const bool f32 = dtype == 1;
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)ld * (f32 ? 4 : 2)};
    cuuint32_t box[2] = {f32 ? 32u : 64u, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1, 1};
    if (fn(map, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base),
           dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
           f32 ? CU_TENSOR_MAP_L2_PROMOTION_NONE : CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return false;
    const int slot = g_map_used < MAP_CACHE ? g_map_used++ : (g_map_next++ % MAP_CACHE);
    g_map_keys[slot] = key;
    g_map_vals[slot] = *map;
    return true;
}
bool gemm_map(CUtensorMap *map, const void *base, long long rows, long long cols, long long ld, int box_rows) {
    return cached_map(map, base, rows, cols, ld, box_rows, 0);
}
// fp32 C [rows][cols], box 32 x 32
bool gemm_map_c(CUtensorMap *map, float *base, long long rows, long long cols, long long ld) {
    return cached_map(map, base, rows, cols, ld, 32, 1);
}

int g_num_sms[64] = {0};

}  // namespace

// Whether the tensor-core kernel can take these operands: TMA needs 16-byte
// aligned bases and row pitches that are multiples of 16 bytes.
bool gemm_tc_ok(const void *A, long long lda, const void *B, long long ldb) {
    return (reinterpret_cast<uintptr_t>(A) & 15u) == 0 && (reinterpret_cast<uintptr_t>(B) & 15u) == 0 &&
           lda % 8 == 0 && ldb % 8 == 0;
}

cudaError_t gemm_bf16(cudaStream_t st, bool ta, bool tb, int M, int N, int K, const void *A, long long lda,
                      const void *B, long long ldb, float *C, long long ldc) {
    if (M <= 0 || N <= 0) return cudaSuccess;
    if (K <= 0) return cudaMemset2DAsync(C, (size_t)ldc * 4, 0, (size_t)N * 4, (size_t)M, st);
    if (!gemm_tc_ok(A, lda, B, ldb)) {
        dim3 grid((unsigned)((N + 31) / 32), (unsigned)((M + 31) / 32));
        gemm_simt_kernel<<<grid, 256, 0, st>>>(static_cast<const __nv_bfloat16 *>(A), lda,
                                               static_cast<const __nv_bfloat16 *>(B), ldb, C, ldc, M, N, K, ta, tb);
        return cudaGetLastError();
    }
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (g_num_sms[dev] == 0) {
        e = cudaDeviceGetAttribute(&g_num_sms[dev], cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(gemm_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)G_SMEM);
        if (e != cudaSuccess) return e;
    }
    const int sms = g_num_sms[dev];
    CUtensorMap ma, mb;
    // A: [M][K] (box 128 rows of M) or [K][M] (box 64 rows of K, two per stage)
    bool okm = ta ? gemm_map(&ma, A, K, M, lda, 64) : gemm_map(&ma, A, M, K, lda, BM);
    // B: [N][K] (box 256 rows of N) or [K][N] (box 64 rows of K, four per stage)
    okm = okm && (tb ? gemm_map(&mb, B, N, K, ldb, BN) : gemm_map(&mb, B, K, N, ldb, 64));
    if (!okm) return cudaErrorInvalidValue;
    GemmArgs g;
    g.C = C;
    g.ldc = ldc;
    g.M = M;
    g.N = N;
    g.K = K;
    g.tiles_m = (M + BM - 1) / BM;
    g.tiles_n = (N + BN - 1) / BN;
    const int nkb = (K + BK - 1) / BK;
    const int tiles = g.tiles_m * g.tiles_n;
    // split K when the output tiles fill less than half of the SMs and each
    // split keeps at least 8 k-blocks
    int splits = 1;
    if (2 * tiles < sms && nkb >= 16) {
        splits = sms / tiles;
        if (splits > nkb / 8) splits = nkb / 8;
        if (splits < 1) splits = 1;
    }
    g.kb_per_split = (nkb + splits - 1) / splits;
    g.splits = (nkb + g.kb_per_split - 1) / g.kb_per_split;
    g.ta = ta;
    g.tb = tb;
    g.vec_ok = (reinterpret_cast<uintptr_t>(C) & 15u) == 0 && ldc % 4 == 0;
    CUtensorMap mc;
    if (g.vec_ok && !gemm_map_c(&mc, C, M, N, ldc)) g.vec_ok = false;
    if (!g.vec_ok) memset(&mc, 0, sizeof(mc));
    if (g.splits > 1) {
        e = cudaMemset2DAsync(C, (size_t)ldc * 4, 0, (size_t)N * 4, (size_t)M, st);
        if (e != cudaSuccess) return e;
    }
    const int work = tiles * g.splits;
    gemm_tc_kernel<<<work < sms ? work : sms, GTHREADS, G_SMEM, st>>>(ma, mb, mc, g);
    return cudaGetLastError();
}

// Reads and clears the flag a GEMM wait sets when it runs out.
int gemm_fault_take() {
    int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_gemm_fault, sizeof(int)) != cudaSuccess) return -1;
    if (v) {
        const int z = 0;
        cudaMemcpyToSymbol(g_gemm_fault, &z, sizeof(int));
    }
    return v;
}

}  // namespace s5
