// s5_forward_tc.cu -- fused S5 forward on the 5th-generation tensor cores.
//
// Layer (review "S5: Simplified State Space Layers for Sequence Modeling", rows
// 1, 3, 4; summary "SIMPLIFIED STATE SPACE LAYERS ...", App. A and App. H):
//   Bu_k = B_bar u_k,  x_k = lambda_bar * x_{k-1} + Bu_k,  y_k = 2 Re(C~ x_k) + D u_k.
//
// A prep kernel writes the bf16 operand images of B_bar and C' into the
// workspace.  Then one persistent CTA per SM claims tiles of 64 tokens of one
// sequence, in order, and runs a warp-specialised pipeline over them:
//   warp 0        TMA: u tile [64 tokens x 128 features] bf16 -> smem (3 stages);
//                 bulk copy of the two weight images at start-up
//   warp 1        tcgen05.mma issuer, driven by whichever input is ready:
//                   GEMM1  Bu^T[2P x 64] = Bs[2P x H] * u^T      (into TMEM)
//                   GEMM2  y^T [H  x 64] = C'[H x 2P] * X^T      (into TMEM)
//   warp 2        TMEM allocation (512 columns: 4 regions of 128)
//   warps 4-7     scan group 0 (even local tiles) } thread = mode = TMEM lane:
//   warps 8-11    scan group 1 (odd local tiles)  } pass 1 folds the tile's 64
//                 steps from zero, publishes the aggregate, decoupled look-back
//                 for the carry, pass 2 reruns from the carry and writes x_k as
//                 bf16 into the GEMM2 operand X [64 x 2P].  Two groups let one
//                 group's look-back overlap the other group's passes.
//   warps 12-15   epilogue: thread = feature = TMEM lane of GEMM2;
//                 y = D2 + D*u, written over u in the stage, TMA store.
// Bs holds B_bar split into real rows (0..P-1) and imaginary rows (P..2P-1);
// C' interleaves (2 Re C~, -2 Im C~) so that K = 2P of GEMM2 pairs with X's
// interleaved (Re x, Im x): sum_k C'[h][k] X[t][k] = 2 Re(C~ x_t)[h].
// Every operand is K-major in the 128-byte-swizzle layout.  Bu and x never
// leave the SM.  All waits are bounded; a wait that runs out latches
// S5_ERR_TIMEOUT, stops the CTA's pipeline, drains its copies and MMAs and
// frees its TMEM.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "s5_internal.cuh"
#include "s5_sm100.cuh"
#include "s5_tc.cuh"

namespace s5 {
using namespace sm100;

namespace {

constexpr int T_TOK = TC_TILE_TOKENS;   // tokens per tile (N of both GEMMs)
constexpr int H_F = 128;                // features
constexpr int P_M = 128;                // stored complex modes
constexpr int STAGES = 3;
constexpr int REGIONS = 4;              // TMEM regions of 128 columns
constexpr int THREADS = 512;
constexpr int W_PROD = 0, W_MMA = 1, W_TMEM = 2, W_SCAN = 4, W_EPI = 12;

constexpr uint32_t BS_BYTES = 2 * 2 * P_M * 128;       // [2 kb][2P rows][128 B]
constexpr uint32_t CP_BYTES = 4 * H_F * 128;           // [4 kb][H rows][128 B]
constexpr uint32_t SM_BS = 0;
constexpr uint32_t SM_CP = SM_BS + BS_BYTES;
constexpr uint32_t SM_U = SM_CP + CP_BYTES;            // [stage][2 kb][64 rows][128 B]
constexpr uint32_t U_STAGE = 2 * T_TOK * 128;
constexpr uint32_t SM_X = SM_U + STAGES * U_STAGE;     // [4 kb][64 rows][128 B]
constexpr uint32_t SM_BAR = SM_X + 4 * T_TOK * 128;
constexpr uint32_t SM_TOTAL = SM_BAR + 512;
constexpr uint32_t SMEM_REQUEST = SM_TOTAL + 1024;     // slack for 1024-B alignment
static_assert(SMEM_REQUEST <= 227 * 1024, "shared memory budget");
static_assert(BS_BYTES + CP_BYTES == 8 * P_M * H_F, "image size");

constexpr unsigned long long PIPE_WAIT_NS = 2000000000ull;   // 2 s per pipeline wait
constexpr unsigned long long DRAIN_WAIT_NS = 200000000ull;   // 0.2 s per teardown wait

struct Bars {
    uint64_t full_u[STAGES], empty_u[STAGES];
    uint64_t tmem_full[REGIONS], tmem_empty[REGIONS], mma2_done[REGIONS];
    uint64_t xready, xfree[2], weights, drain;
    int tile_id[STAGES];
    int n_local;      // tiles this CTA claimed (set once claiming ends), -1 before
    uint32_t tmem_base;
    int abort;
};
static_assert(sizeof(Bars) <= 512, "barrier block");

__device__ __forceinline__ bool aborted(Bars *sb) {
    return *reinterpret_cast<volatile int *>(&sb->abort) != 0;
}
__device__ __forceinline__ void set_abort(Bars *sb, WsHeader *hdr) {
    *reinterpret_cast<volatile int *>(&sb->abort) = 1;
    latch_status(hdr, S5_ERR_TIMEOUT);
}

// Pipeline wait: bounded; gives up at once if another role already aborted.
__device__ __forceinline__ bool pipe_wait(uint64_t *bar, uint32_t parity, Bars *sb, WsHeader *hdr) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = global_ns();
    for (;;) {
        if (aborted(sb)) return false;
        if (mbar_try_wait(bar, parity)) return true;
        if (global_ns() - t0 > PIPE_WAIT_NS) {
            set_abort(sb, hdr);
            return false;
        }
    }
}
// Teardown wait: bounded, ignores the abort flag.
__device__ __forceinline__ bool drain_wait(uint64_t *bar, uint32_t parity) {
    const unsigned long long t0 = global_ns();
    while (!mbar_try_wait(bar, parity))
        if (global_ns() - t0 > DRAIN_WAIT_NS) return false;
    return true;
}

// Tile id of local tile i (-1 when this CTA has no i-th tile, -2 on abort).
__device__ __forceinline__ int wait_tile(int i, Bars *sb, WsHeader *hdr) {
    const int s = i % STAGES;
    const uint32_t par = (i / STAGES) & 1;
    if (mbar_try_wait(&sb->full_u[s], par)) return sb->tile_id[s];
    const unsigned long long t0 = global_ns();
    for (;;) {
        if (aborted(sb)) return -2;
        const int n = *reinterpret_cast<volatile int *>(&sb->n_local);
        if (n >= 0 && i >= n) return -1;
        if (mbar_try_wait(&sb->full_u[s], par)) return sb->tile_id[s];
        if (global_ns() - t0 > PIPE_WAIT_NS) {
            set_abort(sb, hdr);
            return -2;
        }
    }
}

// Byte offset of bf16 element (row, col) in a K-major 128-byte-swizzle region
// whose k-blocks (64 columns each) hold `rows` rows.
__host__ __device__ __forceinline__ uint32_t sw128(uint32_t row, uint32_t col, uint32_t rows) {
    const uint32_t kb = col >> 6, c = col & 63u;
    return kb * rows * 128u + row * 128u + (((c >> 3) ^ (row & 7u)) << 4) + ((c & 7u) << 1);
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

__device__ __forceinline__ float4 ld_volatile_v4(const float4 *p) {
    float4 v;
    asm volatile("ld.volatile.global.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "l"(p));
    return v;
}
__device__ __forceinline__ void st_v4(float4 *p, float a, float b, float c, float d) {
    asm volatile("st.global.cg.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(p), "f"(a), "f"(b), "f"(c),
                 "f"(d)
                 : "memory");
}

__device__ __forceinline__ float2 cpow(float2 a, int n) {
    float2 r = make_float2(1.f, 0.f);
    while (n) {
        if (n & 1) r = cmul(r, a);
        a = cmul(a, a);
        n >>= 1;
    }
    return r;
}

// Carry into tile (b, c) from the per-mode records of tiles (b, c-1), (b, c-2)...
// Each record is one 16-byte word {value.re, value.im, 0, epoch<<2 | state}:
// state 1 = aggregate (end state from zero; the tile's multiplier is
// lambda_bar^64 since only a sequence's last tile can be short), 2 = inclusive
// end state.  Eight predecessors are read per round.
__device__ float2 look_back(const float4 *rec, int B, int b, int c, int m, float2 lbT,
                            unsigned epoch, WsHeader *hdr, unsigned long long limit, int tile) {
    float2 acc = make_float2(0.f, 0.f), mult = make_float2(1.f, 0.f);
    int j = c - 1;
    unsigned long long t0 = 0;
    bool timing = false;
    for (;;) {
        float4 v[8];
#pragma unroll
        for (int w = 0; w < 8; ++w)
            v[w] = (j - w >= 0) ? ld_volatile_v4(rec + ((size_t)(j - w) * B + b) * P_M + m)
                                : make_float4(0.f, 0.f, 0.f, 0.f);
        int used = 0;
        bool done = false;
#pragma unroll
        for (int w = 0; w < 8; ++w) {
            if (done || used != w || j - w < 0) continue;
            const unsigned st = __float_as_uint(v[w].w);
            if ((st >> 2) != epoch || (st & 3u) == 0) continue;
            acc = cfma(mult, make_float2(v[w].x, v[w].y), acc);
            if ((st & 3u) == FLAG_INCL) done = true;
            else {
                mult = cmul(mult, lbT);
                used = w + 1;
            }
        }
        if (done) return acc;
        j -= used;
        if (j < 0) return acc;
        if (used) {
            timing = false;
            continue;
        }
        if (!timing) {
            t0 = global_ns();
            timing = true;
        } else if (global_ns() - t0 > limit) {
            latch_status(hdr, S5_ERR_TIMEOUT);
            atomicCAS(&hdr->timeout_tile, 0u, (unsigned)tile + 1);
            return acc;
        }
        __nanosleep(64);
    }
}

// Loads the Re and Im columns [col, col+16) of this thread's lane.
__device__ __forceinline__ void ld_chunk(uint32_t base, int col, uint32_t (&re)[16],
                                         uint32_t (&im)[16]) {
    tmem_ld16(base + col, re);
    tmem_ld16(base + 64 + col, im);
}

// ---------------------------------------------------------------------------
// Prep: bf16 operand images in the exact byte layout the MMA descriptors read.
// ---------------------------------------------------------------------------
__global__ void weight_images_kernel(const float2 *__restrict__ b_bar, const float2 *__restrict__ c_tilde,
                                     unsigned char *__restrict__ img) {
    const int idx = blockIdx.x * blockDim.x + threadIdx.x;
    if (idx < P_M * H_F / 2) {
        // Bs: rows 0..P-1 = Re B_bar, rows P..2P-1 = Im B_bar, K = H
        const int m = idx / (H_F / 2), h = 2 * (idx % (H_F / 2));
        const float4 v = *reinterpret_cast<const float4 *>(b_bar + (size_t)m * H_F + h);
        *reinterpret_cast<uint32_t *>(img + SM_BS + sw128(m, h, 2 * P_M)) = pack_bf16(v.x, v.z);
        *reinterpret_cast<uint32_t *>(img + SM_BS + sw128(P_M + m, h, 2 * P_M)) = pack_bf16(v.y, v.w);
    } else if (idx < P_M * H_F / 2 + H_F * P_M) {
        // C': row h, columns (2m, 2m+1) = (2 Re C~[h][m], -2 Im C~[h][m]), K = 2P
        const int k = idx - P_M * H_F / 2;
        const int h = k / P_M, m = k % P_M;
        const float2 cv = c_tilde[(size_t)h * P_M + m];
        *reinterpret_cast<uint32_t *>(img + SM_CP + sw128(h, 2 * m, H_F)) =
            pack_bf16(2.f * cv.x, -2.f * cv.y);
    }
}

// ---------------------------------------------------------------------------
// Main kernel.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(THREADS, 1)
fwd_tc_kernel(const __grid_constant__ CUtensorMap tmap_u, const __grid_constant__ CUtensorMap tmap_y,
              const TcArgs args) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char *smem = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    Bars *sb = reinterpret_cast<Bars *>(smem + SM_BAR);
    __shared__ unsigned s_epoch, s_drop;
    __shared__ unsigned long long s_limit;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    WsHeader *hdr = args.ws.hdr;
    float4 *rec = args.ws.agg;
    const int B = args.B, L = args.L;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&sb->full_u[s], 1);
            mbar_init(&sb->empty_u[s], 1);
        }
        for (int r = 0; r < REGIONS; ++r) {
            mbar_init(&sb->tmem_full[r], 1);
            mbar_init(&sb->tmem_empty[r], 4);
            mbar_init(&sb->mma2_done[r], 1);
        }
        mbar_init(&sb->xready, 4);
        mbar_init(&sb->xfree[0], 1);
        mbar_init(&sb->xfree[1], 1);
        mbar_init(&sb->weights, 1);
        mbar_init(&sb->drain, 1);
        sb->n_local = -1;
        sb->abort = 0;
        fence_mbar_init();
        s_epoch = *reinterpret_cast<volatile unsigned *>(&hdr->epoch);
        s_drop = *reinterpret_cast<volatile unsigned *>(&hdr->drop_publish);
        const unsigned lim = *reinterpret_cast<volatile unsigned *>(&hdr->wait_limit_us);
        s_limit = 1000ull * (lim ? lim : 1000000u);
    }
    if (warp == W_TMEM) {
        tmem_alloc(&sb->tmem_base, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sb->tmem_base;
    const unsigned epoch = s_epoch;

    if (warp == W_PROD) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            prefetch_tmap(&tmap_u);
            prefetch_tmap(&tmap_y);
            mbar_arrive_tx(&sb->weights, BS_BYTES + CP_BYTES);
            bulk_load(smem + SM_BS, args.ws.wimg + SM_BS, BS_BYTES, &sb->weights);
            bulk_load(smem + SM_CP, args.ws.wimg + SM_CP, CP_BYTES, &sb->weights);
            int last_issue[STAGES] = {-1, -1, -1};
            int i = 0;
            for (;; ++i) {
                const int s = i % STAGES;
                if (i >= STAGES && !pipe_wait(&sb->empty_u[s], ((i / STAGES) - 1) & 1, sb, hdr)) break;
                const int tile = (int)atomicAdd(&hdr->tile_counter, 1u);
                if (tile >= args.ntiles) break;
                sb->tile_id[s] = tile;
                const int b = tile % B, c = tile / B;
                unsigned char *dst = smem + SM_U + s * U_STAGE;
                mbar_arrive_tx(&sb->full_u[s], U_STAGE);
                tma_load_3d(dst, &tmap_u, 0, c * T_TOK, b, &sb->full_u[s]);
                tma_load_3d(dst + T_TOK * 128, &tmap_u, 64, c * T_TOK, b, &sb->full_u[s]);
                last_issue[s] = i;
            }
            // consumers waiting for local tile i (never loaded) see the end here
            *reinterpret_cast<volatile int *>(&sb->n_local) = i;
            // copies still in flight must land before the CTA exits
            drain_wait(&sb->weights, 0);
            for (int s = 0; s < STAGES; ++s)
                if (last_issue[s] >= 0) drain_wait(&sb->full_u[s], (last_issue[s] / STAGES) & 1);
        }
    } else if (warp == W_MMA) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            const uint32_t idesc = idesc_bf16_f32(128, T_TOK);
            const uint32_t bs = smem_addr(smem + SM_BS), cp = smem_addr(smem + SM_CP);
            const uint32_t xs = smem_addr(smem + SM_X);
            bool ok = pipe_wait(&sb->weights, 0, sb, hdr);
            int g1 = 0, g2 = 0;          // next tile for GEMM1 / GEMM2
            int n_end = -1;              // tiles of this CTA, once known
            unsigned long long t0 = global_ns();
            while (ok) {
                bool progress = false;
                // GEMM1 of tile g1: u tile landed and its TMEM region is free
                if (n_end < 0 || g1 < n_end) {
                    const int s = g1 % STAGES, r = g1 % REGIONS;
                    const int n = *reinterpret_cast<volatile int *>(&sb->n_local);
                    if (n >= 0 && g1 >= n) {
                        n_end = n;
                    } else if (mbar_test_wait(&sb->full_u[s], (g1 / STAGES) & 1) &&
                               (g1 < REGIONS ||
                                mbar_test_wait(&sb->tmem_empty[r], ((g1 / REGIONS) - 1) & 1))) {
                        tc_fence_after();
                        const uint32_t ub = smem_addr(smem + SM_U + s * U_STAGE);
                        for (int mb = 0; mb < 2; ++mb)
                            for (int k = 0; k < H_F / 16; ++k)
                                mma_bf16(tmem + (uint32_t)r * 128u + (uint32_t)mb * 64u,
                                         sw128_kmajor_desc(bs + (k >> 2) * (2 * P_M * 128) +
                                                           mb * (P_M * 128) + (k & 3) * 32),
                                         sw128_kmajor_desc(ub + (k >> 2) * (T_TOK * 128) + (k & 3) * 32),
                                         idesc, k > 0);
                        mma_commit(&sb->tmem_full[r]);
                        ++g1;
                        progress = true;
                    }
                }
                // GEMM2 of tile g2: its scan wrote X
                if (g2 < g1 && mbar_test_wait(&sb->xready, g2 & 1)) {
                    tc_fence_after();
                    const uint32_t d = tmem + (uint32_t)(g2 % REGIONS) * 128u;
                    for (int k = 0; k < 2 * P_M / 16; ++k)
                        mma_bf16(d, sw128_kmajor_desc(cp + (k >> 2) * (H_F * 128) + (k & 3) * 32),
                                 sw128_kmajor_desc(xs + (k >> 2) * (T_TOK * 128) + (k & 3) * 32),
                                 idesc, k > 0);
                    mma_commit(&sb->mma2_done[g2 % REGIONS]);
                    mma_commit(&sb->xfree[g2 & 1]);
                    ++g2;
                    progress = true;
                }
                if (n_end >= 0 && g2 >= n_end) break;
                if (progress) {
                    t0 = global_ns();
                } else if (aborted(sb)) {
                    break;
                } else if (global_ns() - t0 > PIPE_WAIT_NS) {
                    set_abort(sb, hdr);
                    break;
                }
            }
            // every MMA issued must complete before TMEM is freed
            mma_commit(&sb->drain);
            drain_wait(&sb->drain, 0);
        }
    } else if (warp >= W_SCAN && warp < W_SCAN + 8) {
        // ------------------------------------------------------------ scan groups
        const int grp = (warp - W_SCAN) >> 2;   // 0: even local tiles, 1: odd
        const int qd = (warp - W_SCAN) & 3;     // TMEM lane quarter
        const int m = 32 * qd + lane;
        const float2 lb = args.lambda_bar[m];
        float2 lbT = lb;
        for (int e = 1; e < T_TOK; e <<= 1) lbT = cmul(lbT, lbT);
        const uint32_t lane_base = tmem + ((uint32_t)(32 * qd) << 16);
        unsigned char *xw = smem + SM_X + qd * (T_TOK * 128);
        const uint32_t xcol = (uint32_t)lane * 4u;   // byte of (Re, Im) in this warp's k-block row
        for (int i = grp;; i += 2) {
            const int tile = wait_tile(i, sb, hdr);
            if (tile < 0) break;
            const int b = tile % B, c = tile / B;
            const int Tc = min(T_TOK, L - c * T_TOK);
            const int r = i % REGIONS;
            if (!pipe_wait(&sb->tmem_full[r], (i / REGIONS) & 1, sb, hdr)) break;
            tc_fence_after();
            const uint32_t col0 = lane_base + (uint32_t)r * 128u;

            // pass 1: end state of the tile from a zero start
            float2 E = make_float2(0.f, 0.f);
            {
                uint32_t re[16], im[16];
                ld_chunk(col0, 0, re, im);
                tmem_wait_ld();
#pragma unroll 1
                for (int ch = 0; ch < T_TOK / 16; ++ch) {
                    if (ch * 16 >= Tc) break;
                    float2 v[16];
#pragma unroll
                    for (int k = 0; k < 16; ++k)
                        v[k] = make_float2(__uint_as_float(re[k]), __uint_as_float(im[k]));
                    if ((ch + 1) * 16 < Tc) ld_chunk(col0, (ch + 1) * 16, re, im);
                    const int n = Tc - ch * 16;
#pragma unroll
                    for (int k = 0; k < 16; ++k)
                        if (k < n) E = cfma(lb, E, v[k]);
                    tmem_wait_ld();
                }
            }
            const float2 A = (Tc == T_TOK) ? lbT : cpow(lb, Tc);
            const bool publish = s_drop != (unsigned)(tile + 1);
            float4 *my = rec + (size_t)tile * P_M + m;
            float2 carry = make_float2(0.f, 0.f);
            if (c == 0) {
                if (args.x0) carry = args.x0[(size_t)b * P_M + m];
            } else {
                if (publish) st_v4(my, E.x, E.y, 0.f, __uint_as_float((epoch << 2) | FLAG_AGG));
                carry = look_back(rec, B, b, c, m, lbT, epoch, hdr, s_limit, tile);
            }
            const float2 inc = cfma(A, carry, E);
            if (publish) st_v4(my, inc.x, inc.y, 0.f, __uint_as_float((epoch << 2) | FLAG_INCL));

            // pass 2: states from the carry, written as the bf16 GEMM2 operand
            if (i >= 1 && !pipe_wait(&sb->xfree[(i - 1) & 1], ((i - 1) >> 1) & 1, sb, hdr)) break;
            float2 x = carry;
            {
                uint32_t re[16], im[16];
                ld_chunk(col0, 0, re, im);
                tmem_wait_ld();
#pragma unroll 1
                for (int ch = 0; ch < T_TOK / 16; ++ch) {
                    const bool live = ch * 16 < Tc;
                    float2 v[16];
#pragma unroll
                    for (int k = 0; k < 16; ++k)
                        v[k] = make_float2(__uint_as_float(re[k]), __uint_as_float(im[k]));
                    if ((ch + 1) * 16 < Tc) ld_chunk(col0, (ch + 1) * 16, re, im);
#pragma unroll
                    for (int k = 0; k < 16; ++k) {
                        const int t = ch * 16 + k;
                        uint32_t pv = 0;
                        if (live && t < Tc) {
                            x = cfma(lb, x, v[k]);
                            pv = pack_bf16(x.x, x.y);
                        }
                        *reinterpret_cast<uint32_t *>(xw + t * 128 + (((xcol >> 4) ^ (uint32_t)(t & 7)) << 4) +
                                                      (xcol & 15u)) = pv;
                    }
                    tmem_wait_ld();
                }
            }
            if (c == args.nchunks - 1 && args.x_last) args.x_last[(size_t)b * P_M + m] = x;
            fence_proxy_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&sb->xready);
        }
    } else if (warp >= W_EPI && warp < W_EPI + 4) {
        // ------------------------------------------------------------ epilogue
        const int qd = warp - W_EPI;
        const int h = 32 * qd + lane;
        const float dh = args.d[h];
        const uint32_t lane_base = tmem + ((uint32_t)(32 * qd) << 16);
        const uint32_t hkb = (uint32_t)h >> 6, hc = (uint32_t)h & 63u;
        const bool leader = (threadIdx.x == W_EPI * 32);
        for (int i = 0;; ++i) {
            const int tile = wait_tile(i, sb, hdr);
            if (tile < 0) break;
            const int s = i % STAGES, r = i % REGIONS;
            if (!pipe_wait(&sb->mma2_done[r], (i / REGIONS) & 1, sb, hdr)) break;
            tc_fence_after();
            uint32_t yv[T_TOK];
#pragma unroll
            for (int ch = 0; ch < T_TOK / 16; ++ch)
                tmem_ld16(lane_base + (uint32_t)r * 128u + ch * 16,
                          *reinterpret_cast<uint32_t(*)[16]>(&yv[ch * 16]));
            tmem_wait_ld();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&sb->tmem_empty[r]);
            unsigned char *stage = smem + SM_U + s * U_STAGE + hkb * (T_TOK * 128);
#pragma unroll
            for (int t0 = 0; t0 < T_TOK; t0 += 16) {
                __nv_bfloat16 uvals[16];
#pragma unroll
                for (int k = 0; k < 16; ++k) {
                    const int t = t0 + k;
                    uvals[k] = *reinterpret_cast<const __nv_bfloat16 *>(
                        stage + t * 128 + (((hc >> 3) ^ (uint32_t)(t & 7)) << 4) + ((hc & 7u) << 1));
                }
#pragma unroll
                for (int k = 0; k < 16; ++k) {
                    const int t = t0 + k;
                    *reinterpret_cast<__nv_bfloat16 *>(
                        stage + t * 128 + (((hc >> 3) ^ (uint32_t)(t & 7)) << 4) + ((hc & 7u) << 1)) =
                        __float2bfloat16_rn(fmaf(dh, __bfloat162float(uvals[k]), __uint_as_float(yv[t])));
                }
            }
            fence_proxy_async_smem();
            named_bar_sync(1, 128);
            if (leader) {
                const int b = tile % B, c = tile / B;
                unsigned char *src = smem + SM_U + s * U_STAGE;
                tma_store_3d(&tmap_y, src, 0, c * T_TOK, b);
                tma_store_3d(&tmap_y, src + T_TOK * 128, 64, c * T_TOK, b);
                bulk_commit();
                bulk_wait_read_all();
                mbar_arrive(&sb->empty_u[s]);
            }
        }
        if (leader) bulk_wait_all();
    }

    // ---------------------------------------------------------------- teardown
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == W_TMEM) tmem_dealloc(tmem, 512);
    if (threadIdx.x == 0) {
        __threadfence();
        const unsigned prev = atomicAdd(&hdr->done_counter, 1u);
        if (prev == gridDim.x - 1) {
            hdr->tile_counter = 0;
            hdr->done_counter = 0;
            hdr->epoch = (s_epoch + 1) & 0x3FFFFFFFu;
            __threadfence();
        }
    }
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    return fn;
}

// [B][L][128] bf16, boxes of 64 features x 64 tokens x 1 sequence, 128-byte swizzle;
// rows past L read as zero and are not written.
bool make_map(CUtensorMap *map, const void *base, int B, int L) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {(cuuint64_t)H_F, (cuuint64_t)L, (cuuint64_t)B};
    cuuint64_t strides[2] = {(cuuint64_t)H_F * 2, (cuuint64_t)L * H_F * 2};
    cuuint32_t box[3] = {64, (cuuint32_t)T_TOK, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides,
                    box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

}  // namespace

bool tc_supported(int H, int P, bool u_bf16, bool y_bf16, bool proj_bf16) {
    return H == H_F && P == P_M && u_bf16 && y_bf16 && proj_bf16;
}

cudaError_t launch_forward_tc(const TcArgs &a, const void *u, void *y, cudaStream_t st,
                              int num_sms) {
    CUtensorMap mu, my;
    if (!make_map(&mu, u, a.B, a.L) || !make_map(&my, y, a.B, a.L)) return cudaErrorInvalidValue;
    const int words = P_M * H_F / 2 + H_F * P_M;
    weight_images_kernel<<<(words + 255) / 256, 256, 0, st>>>(a.b_bar, a.c_tilde, a.ws.wimg);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(fwd_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)SMEM_REQUEST);
    if (e != cudaSuccess) return e;
    int grid = num_sms < a.ntiles ? num_sms : a.ntiles;
    fwd_tc_kernel<<<grid, THREADS, SMEM_REQUEST, st>>>(mu, my, a);
    return cudaGetLastError();
}

}  // namespace s5
