// s5_forward_tc.cu -- fused S5 forward on the 5th-generation tensor cores.
//
// Layer (review "S5: Simplified State Space Layers for Sequence Modeling", rows
// 1, 3, 4; summary "SIMPLIFIED STATE SPACE LAYERS ...", App. A and App. H):
//   Bu_k = B_bar u_k,  x_k = lambda_bar * x_{k-1} + Bu_k,  y_k = 2 Re(C~ x_k) + D u_k.
//
// A prep kernel writes the bf16 operand images of B_bar and C' into the
// workspace.  Then one persistent CTA per SM (a cooperative launch, so every
// CTA is resident) takes the tiles k, k+G, k+2G, ... of 64 tokens (G = grid):
// all CTAs work through the same "wave" of G tiles at the same time, so a
// tile's predecessors in its sequence are same-wave tiles being scanned
// concurrently, and the look-back waits on no other CTA's queue.  Each CTA
// runs a warp-specialised pipeline over its tiles:
//   warp 0        TMA: u tile [64 tokens x 128 features] bf16 -> smem (4 stages);
//                 bulk copy of the two weight images at start-up
//   warp 1        tcgen05.mma issuer, driven by whichever input is ready:
//                   GEMM1  Bu^T[2P x 64] = Bs[2P x H] * u^T      (into TMEM)
//                   GEMM2  y^T [H  x 64] = C'[H x 2P] * X^T      (into TMEM)
//   warp 2        TMEM allocation (512 columns: 4 regions of 128)
//   warps 4-7     scan: thread = mode = TMEM lane, one tile ahead:
//                 pass 1 of tile i+1 folds its 64 steps from zero and
//                 publishes the aggregate; the look-back loads for tile i+1
//                 are issued; pass 2 of tile i reruns from its carry (two
//                 interleaved 32-step chains) and writes x_k as bf16 into the
//                 GEMM2 operand X [64 x 2P]; then the look-back of tile i+1
//                 resolves and its inclusive state is published.
//   warps 8-11    epilogue: thread = feature = TMEM lane of GEMM2;
//                 y = D2 + D*u with u read from the stage (the stage is free
//                 once GEMM1 and the epilogue have read it), stored as bf16
//                 with one 64-byte segment per warp and token.
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
constexpr int STAGES = 4;
constexpr int REGIONS = 4;              // TMEM regions of 128 columns
constexpr int THREADS = 384;
constexpr int W_PROD = 0, W_MMA = 1, W_TMEM = 2, W_SCAN = 4, W_EPI = 8;

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
    uint64_t xready, xfree, weights, drain;
    int n_local;      // tiles of this CTA
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

// Pipeline wait: bounded; gives up once another role has aborted.  The
// waiting warp sleeps in hardware (suspend-time hint) until the phase
// completes, so it takes no issue slots from the warps sharing its SM
// sub-partition.
constexpr uint32_t SLEEP_HINT_NS = 1000000;   // re-check abort/limits every 1 ms
__device__ __forceinline__ bool pipe_wait(uint64_t *bar, uint32_t parity, Bars *sb, WsHeader *hdr) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = global_ns();
    for (;;) {
        if (mbar_try_wait_sleep(bar, parity, SLEEP_HINT_NS)) return true;
        if (aborted(sb)) return false;
        if (global_ns() - t0 > PIPE_WAIT_NS) {
            set_abort(sb, hdr);
            return false;
        }
    }
}
// Teardown wait: bounded, ignores the abort flag.
__device__ __forceinline__ bool drain_wait(uint64_t *bar, uint32_t parity) {
    const unsigned long long t0 = global_ns();
    while (!mbar_try_wait_sleep(bar, parity, SLEEP_HINT_NS))
        if (global_ns() - t0 > DRAIN_WAIT_NS) return false;
    return true;
}

// Tile id of local tile i once its u tile has landed (-1 when this CTA has
// no i-th tile, -2 on abort).
__device__ __forceinline__ int wait_tile(int i, Bars *sb, WsHeader *hdr) {
    if (i >= sb->n_local) return -1;
    if (!pipe_wait(&sb->full_u[i % STAGES], (i / STAGES) & 1, sb, hdr)) return -2;
    return (int)blockIdx.x + i * (int)gridDim.x;
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

// Carry records are read and written with GPU-scope relaxed 16-byte accesses
// (a record is written whole, so a reader sees its state and value together;
// system-scope accesses would be needlessly slow on a host-coherent GPU).
__device__ __forceinline__ float4 ld_record(const float4 *p) {
    float4 v;
    asm volatile("ld.relaxed.gpu.global.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "l"(p)
                 : "memory");
    return v;
}
__device__ __forceinline__ void st_record(float4 *p, float a, float b, float c, float d) {
    asm volatile("st.relaxed.gpu.global.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(p), "f"(a), "f"(b),
                 "f"(c), "f"(d)
                 : "memory");
}

__device__ __forceinline__ void sts32(uint32_t addr, uint32_t v) {
    asm volatile("st.shared.b32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}
__device__ __forceinline__ uint32_t lds16(uint32_t addr) {
    unsigned short v;
    asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(addr) : "memory");
    return v;
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
// end state.  LB_WIN predecessors are read per round.
constexpr int LB_WIN = 8;    // records loaded an iteration ahead
constexpr int LB_WIN2 = 12;  // records loaded when the look-back resolves (together: 20,
                             // a whole wave of one sequence, G / B = 19 chunks, in one round)
// Loads the records of chunks j, j-1, ..., j-LB_WIN+1 of this mode.
__device__ __forceinline__ void lb_issue(float4 (&v)[LB_WIN], const float4 *col, size_t stride, int j) {
    const float4 *pj = col + (size_t)j * stride;
#pragma unroll
    for (int w = 0; w < LB_WIN; ++w)
        v[w] = (j - w >= 0) ? ld_record(pj - (size_t)w * stride) : make_float4(0.f, 0.f, 0.f, 0.f);
}

// Folds one window of records into (acc, mult), newest first.  Returns 1 when
// an inclusive record ended the chain, 0 when the window was used up, -1 when
// a record was not ready (j then names the first record still needed).
template <int W>
__device__ __forceinline__ int lb_fold(const float4 (&v)[W], int &j, float2 &acc, float2 &mult,
                                       float2 lbT, unsigned agg, unsigned incl) {
#pragma unroll
    for (int w = 0; w < W; ++w) {
        if (j < 0) return 0;
        const unsigned st = __float_as_uint(v[w].w);
        const bool is_incl = st == incl;
        if (!(is_incl || st == agg)) return -1;
        acc = cfma(mult, make_float2(v[w].x, v[w].y), acc);
        if (is_incl) return 1;
        mult = cmul(mult, lbT);
        --j;
    }
    return 0;
}

// Carry of chunk j+1: folds the records of chunks j, j-1, ... until an
// inclusive one.  v holds the LB_WIN records from chunk j down, loaded
// earlier by lb_issue; the next LB_WIN2 are loaded on entry so that their
// latency overlaps the first fold, and further windows are loaded as needed.
__device__ float2 lb_finish(float4 (&v)[LB_WIN], const float4 *col, size_t stride, int j,
                            float2 lbT, unsigned epoch, WsHeader *hdr, unsigned long long limit,
                            int tile) {
    float2 acc = make_float2(0.f, 0.f), mult = make_float2(1.f, 0.f);
    const unsigned agg = (epoch << 2) | FLAG_AGG, incl = (epoch << 2) | FLAG_INCL;
    float4 v2[LB_WIN2];
    {
        const float4 *pj = col + (size_t)(j - LB_WIN) * stride;
#pragma unroll
        for (int w = 0; w < LB_WIN2; ++w)
            v2[w] = (j - LB_WIN - w >= 0) ? ld_record(pj - (size_t)w * stride)
                                          : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    int rc = lb_fold<LB_WIN>(v, j, acc, mult, lbT, agg, incl);
    if (rc == 1) return acc;
    if (rc == 0) {
        rc = lb_fold<LB_WIN2>(v2, j, acc, mult, lbT, agg, incl);
        if (rc == 1) return acc;
    }
    // slow path: chains longer than one wave, or records not yet published
    unsigned long long t0 = 0;
    bool timing = false;
    int last_j = j;
    for (;;) {
        if (j < 0) return acc;
        lb_issue(v, col, stride, j);
        rc = lb_fold<LB_WIN>(v, j, acc, mult, lbT, agg, incl);
        if (rc == 1) return acc;
        if (j < last_j) {
            timing = false;
            last_j = j;
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
// Scan passes over one tile of this thread's mode (TMEM lane): D1 columns
// [col0, col0+64) hold Re(Bu_t), [col0+64, col0+128) hold Im(Bu_t).
// ---------------------------------------------------------------------------
struct ScanConsts {
    float2 lb, lb8, lb16, lb32, lb64;   // lambda_bar and its powers
};

__device__ __forceinline__ float2 tmem_pair(const uint32_t (&re)[16], const uint32_t (&im)[16], int k) {
    return make_float2(__uint_as_float(re[k]), __uint_as_float(im[k]));
}

// Full tile: end state from zero over tokens 0..31 (elo) and 0..63 (returned),
// as two interleaved 32-step chains over tokens 0..31 and 32..63.
__device__ __forceinline__ float2 pass1_full(uint32_t col0, const ScanConsts &k, float2 &elo) {
    float2 ea = make_float2(0.f, 0.f), ez = make_float2(0.f, 0.f);
#pragma unroll 1
    for (int c8 = 0; c8 < 4; ++c8) {
        uint32_t ra[8], ia[8], rz[8], iz[8];
        tmem_ld8(col0 + c8 * 8, ra);
        tmem_ld8(col0 + 64 + c8 * 8, ia);
        tmem_ld8(col0 + 32 + c8 * 8, rz);
        tmem_ld8(col0 + 96 + c8 * 8, iz);
        tmem_wait_ld();
#pragma unroll
        for (int t = 0; t < 8; ++t) {
            ea = cfma(k.lb, ea, make_float2(__uint_as_float(ra[t]), __uint_as_float(ia[t])));
            ez = cfma(k.lb, ez, make_float2(__uint_as_float(rz[t]), __uint_as_float(iz[t])));
        }
    }
    elo = ea;
    return cfma(k.lb32, ea, ez);
}

// Short tile (Tc < 64): end state from zero over its Tc tokens.
__device__ float2 pass1_short(uint32_t col0, int Tc, float2 lb) {
    float2 e = make_float2(0.f, 0.f);
#pragma unroll 1
    for (int ch = 0; ch * 16 < Tc; ++ch) {
        uint32_t re[16], im[16];
        ld_chunk(col0, ch * 16, re, im);
        tmem_wait_ld();
        const int n = Tc - ch * 16;
#pragma unroll
        for (int t = 0; t < 16; ++t)
            if (t < n) e = cfma(lb, e, tmem_pair(re, im, t));
    }
    return e;
}

// Full tile: states from the carry as two interleaved 32-step chains (the
// second starts from lambda_bar^32 carry + elo), each written as bf16 (Re, Im)
// into row t of X.  Returns the state after token 63.
__device__ __forceinline__ float2 pass2_full(uint32_t col0, const uint32_t (&xb)[8], const ScanConsts &k,
                                             float2 carry, float2 elo) {
    float2 xa = carry, xz = cfma(k.lb32, carry, elo);
#pragma unroll 1   // rolled: keeps the scan warps within their register budget
    for (int c8 = 0; c8 < 4; ++c8) {
        // tokens 8*c8 .. +7 (chain a) and 32 + 8*c8 .. +7 (chain z)
        uint32_t ra[8], ia[8], rz[8], iz[8];
        tmem_ld8(col0 + c8 * 8, ra);
        tmem_ld8(col0 + 64 + c8 * 8, ia);
        tmem_ld8(col0 + 32 + c8 * 8, rz);
        tmem_ld8(col0 + 96 + c8 * 8, iz);
        tmem_wait_ld();
#pragma unroll
        for (int t = 0; t < 8; ++t) {
            xa = cfma(k.lb, xa, make_float2(__uint_as_float(ra[t]), __uint_as_float(ia[t])));
            xz = cfma(k.lb, xz, make_float2(__uint_as_float(rz[t]), __uint_as_float(iz[t])));
            // row 8*c8 + t lives at xb[t] + c8 * 1024; row 32 + 8*c8 + t at xb[t] + (4 + c8) * 1024
            sts32(xb[t] + (uint32_t)c8 * 1024u, pack_bf16(xa.x, xa.y));
            sts32(xb[t] + (uint32_t)(4 + c8) * 1024u, pack_bf16(xz.x, xz.y));
        }
    }
    return xz;
}

// Short tile: sequential states; rows past Tc are written as zeros.
__device__ float2 pass2_short(uint32_t col0, const uint32_t (&xb)[8], float2 lb, float2 x, int Tc) {
#pragma unroll 1
    for (int ch = 0; ch < T_TOK / 16; ++ch) {
        uint32_t re[16], im[16];
        const bool live = ch * 16 < Tc;
        if (live) {
            ld_chunk(col0, ch * 16, re, im);
            tmem_wait_ld();
        }
#pragma unroll
        for (int t = 0; t < 16; ++t) {
            uint32_t pv = 0;
            if (live && ch * 16 + t < Tc) {
                x = cfma(lb, x, tmem_pair(re, im, t));
                pv = pack_bf16(x.x, x.y);
            }
            sts32(xb[t & 7] + (uint32_t)((ch * 16 + t) >> 3) * 1024u, pv);
        }
    }
    return x;
}

// One tile of the scan stage.
struct ScanTile {
    int tile, b, c, Tc, r;
    float2 E, elo, carry;
    bool pending;   // look-back still to resolve
};

// Everything the scan warps need that does not change from tile to tile.
struct ScanCtx {
    ScanConsts kc;
    uint32_t lane_base;
    float4 *rec;
    const float2 *x0;
    size_t stride;
    int B, L, m;
    unsigned epoch, drop, agg_word, incl_word;
    unsigned long long limit;
    WsHeader *hdr;
};

// Pass 1 of a tile whose D1 has landed; publishes its aggregate (or, for a
// sequence's first chunk, its inclusive state) and issues its look-back loads.
__device__ __forceinline__ void scan_front(const ScanCtx &x, ScanTile &T) {
    const uint32_t col0 = x.lane_base + (uint32_t)T.r * 128u;
    T.elo = make_float2(0.f, 0.f);
    T.E = (T.Tc == T_TOK) ? pass1_full(col0, x.kc, T.elo) : pass1_short(col0, T.Tc, x.kc.lb);
    const bool publish = x.drop != (unsigned)(T.tile + 1);
    float4 *my = x.rec + (size_t)T.tile * P_M + x.m;
    if (T.c == 0) {
        T.carry = x.x0 ? x.x0[(size_t)T.b * P_M + x.m] : make_float2(0.f, 0.f);
        const float2 A = (T.Tc == T_TOK) ? x.kc.lb64 : cpow(x.kc.lb, T.Tc);
        const float2 inc = cfma(A, T.carry, T.E);
        if (publish) st_record(my, inc.x, inc.y, 0.f, __uint_as_float(x.incl_word));
        T.pending = false;
    } else {
        if (publish) st_record(my, T.E.x, T.E.y, 0.f, __uint_as_float(x.agg_word));
        T.pending = true;
    }
}

// Issues the first window of look-back loads of a pending tile.
__device__ __forceinline__ void scan_issue(const ScanCtx &x, const ScanTile &T, float4 (&v)[LB_WIN]) {
    lb_issue(v, x.rec + (size_t)T.b * P_M + x.m, x.stride, T.c - 1);
}

// Completes the look-back of a tile and publishes its inclusive state.
__device__ __forceinline__ void scan_resolve(const ScanCtx &x, ScanTile &T, float4 (&v)[LB_WIN]) {
    T.carry = lb_finish(v, x.rec + (size_t)T.b * P_M + x.m, x.stride, T.c - 1, x.kc.lb64, x.epoch,
                        x.hdr, x.limit, T.tile);
    const float2 A = (T.Tc == T_TOK) ? x.kc.lb64 : cpow(x.kc.lb, T.Tc);
    const float2 inc = cfma(A, T.carry, T.E);
    if (x.drop != (unsigned)(T.tile + 1))
        st_record(x.rec + (size_t)T.tile * P_M + x.m, inc.x, inc.y, 0.f, __uint_as_float(x.incl_word));
    T.pending = false;
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
fwd_tc_kernel(const __grid_constant__ CUtensorMap tmap_u, const TcArgs args) {
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
            mbar_init(&sb->empty_u[s], 5);   // GEMM1 commit + 4 epilogue warps
        }
        for (int r = 0; r < REGIONS; ++r) {
            mbar_init(&sb->tmem_full[r], 1);
            mbar_init(&sb->tmem_empty[r], 4);
            mbar_init(&sb->mma2_done[r], 1);
        }
        mbar_init(&sb->xready, 4);
        mbar_init(&sb->xfree, 1);
        mbar_init(&sb->weights, 1);
        mbar_init(&sb->drain, 1);
        sb->n_local = args.ntiles > (int)blockIdx.x
                          ? (args.ntiles - (int)blockIdx.x + (int)gridDim.x - 1) / (int)gridDim.x
                          : 0;
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
            mbar_arrive_tx(&sb->weights, BS_BYTES + CP_BYTES);
            bulk_load(smem + SM_BS, args.ws.wimg + SM_BS, BS_BYTES, &sb->weights);
            bulk_load(smem + SM_CP, args.ws.wimg + SM_CP, CP_BYTES, &sb->weights);
            int last_issue[STAGES];
            for (int s = 0; s < STAGES; ++s) last_issue[s] = -1;
            const int n_local = sb->n_local;
            for (int i = 0; i < n_local; ++i) {
                const int s = i % STAGES;
                if (i >= STAGES && !pipe_wait(&sb->empty_u[s], ((i / STAGES) - 1) & 1, sb, hdr)) break;
                const int tile = (int)blockIdx.x + i * (int)gridDim.x;
                const int b = tile % B, c = tile / B;
                unsigned char *dst = smem + SM_U + s * U_STAGE;
                mbar_arrive_tx(&sb->full_u[s], U_STAGE);
                tma_load_3d(dst, &tmap_u, 0, c * T_TOK, b, &sb->full_u[s]);
                tma_load_3d(dst + T_TOK * 128, &tmap_u, 64, c * T_TOK, b, &sb->full_u[s]);
                last_issue[s] = i;
            }
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
            const int n_end = sb->n_local;
            unsigned long long t0 = global_ns();
            while (ok) {
                bool progress = false;
                // GEMM1 of tile g1: u tile landed and its TMEM region is free
                if (g1 < n_end) {
                    const int s = g1 % STAGES, r = g1 % REGIONS;
                    if (mbar_test_wait(&sb->full_u[s], (g1 / STAGES) & 1) &&
                               (g1 < REGIONS ||
                                mbar_test_wait(&sb->tmem_empty[r], ((g1 / REGIONS) - 1) & 1))) {
                        tc_fence_after();
                        const uint32_t ub = smem_addr(smem + SM_U + s * U_STAGE);
                        // rolled loops: descriptors are rebuilt per MMA rather than
                        // hoisted into (many) registers
#pragma unroll 1
                        for (int mb = 0; mb < 2; ++mb)
#pragma unroll 1
                            for (int k = 0; k < H_F / 16; ++k)
                                mma_bf16(tmem + (uint32_t)r * 128u + (uint32_t)mb * 64u,
                                         sw128_kmajor_desc(bs + (k >> 2) * (2 * P_M * 128) +
                                                           mb * (P_M * 128) + (k & 3) * 32),
                                         sw128_kmajor_desc(ub + (k >> 2) * (T_TOK * 128) + (k & 3) * 32),
                                         idesc, k > 0);
                        mma_commit(&sb->tmem_full[r]);
                        mma_commit(&sb->empty_u[s]);
                        ++g1;
                        progress = true;
                    }
                }
                // GEMM2 of tile g2: its scan wrote X
                if (g2 < g1 && mbar_test_wait(&sb->xready, g2 & 1)) {
                    tc_fence_after();
                    const uint32_t d = tmem + (uint32_t)(g2 % REGIONS) * 128u;
#pragma unroll 1
                    for (int k = 0; k < 2 * P_M / 16; ++k)
                        mma_bf16(d, sw128_kmajor_desc(cp + (k >> 2) * (H_F * 128) + (k & 3) * 32),
                                 sw128_kmajor_desc(xs + (k >> 2) * (T_TOK * 128) + (k & 3) * 32),
                                 idesc, k > 0);
                    mma_commit(&sb->mma2_done[g2 % REGIONS]);
                    mma_commit(&sb->xfree);
                    ++g2;
                    progress = true;
                }
                if (g2 >= n_end) break;
                if (progress) {
                    t0 = global_ns();
                } else if (aborted(sb)) {
                    break;
                } else if (global_ns() - t0 > PIPE_WAIT_NS) {
                    set_abort(sb, hdr);
                    break;
                } else {
                    // yield the issue slots of this SM sub-partition to the
                    // scan and epilogue warps that share it
                    __nanosleep(64);
                }
            }
            // every MMA issued must complete before TMEM is freed
            mma_commit(&sb->drain);
            drain_wait(&sb->drain, 0);
        }
    } else if (warp >= W_SCAN && warp < W_SCAN + 4) {
        // ------------------------------------------------------------ scan
        const int qd = warp - W_SCAN;           // TMEM lane quarter
        const int m = 32 * qd + lane;
        ScanConsts kc;
        kc.lb = args.lambda_bar[m];
        kc.lb8 = cpow(kc.lb, 8);
        kc.lb16 = cmul(kc.lb8, kc.lb8);
        kc.lb32 = cmul(kc.lb16, kc.lb16);
        kc.lb64 = cmul(kc.lb32, kc.lb32);
        const uint32_t lane_base = tmem + ((uint32_t)(32 * qd) << 16);
        const uint32_t xcol = (uint32_t)lane * 4u;   // byte of (Re, Im) in this warp's k-block row
        // shared address of (row q, this lane's column) in each swizzle phase q;
        // row t lives at xb[t & 7] + (t >> 3) * 1024
        uint32_t xb[8];
#pragma unroll
        for (int q = 0; q < 8; ++q)
            xb[q] = smem_addr(smem + SM_X + qd * (T_TOK * 128)) + 128u * q +
                    ((((xcol >> 4) ^ (uint32_t)q)) << 4) + (xcol & 15u);
        ScanCtx cx;
        cx.kc = kc;
        cx.lane_base = lane_base;
        cx.rec = rec;
        cx.x0 = args.x0;
        cx.stride = (size_t)B * P_M;
        cx.B = B;
        cx.L = L;
        cx.m = m;
        cx.epoch = epoch;
        cx.drop = s_drop;
        cx.agg_word = (epoch << 2) | FLAG_AGG;
        cx.incl_word = (epoch << 2) | FLAG_INCL;
        cx.limit = s_limit;
        cx.hdr = hdr;
        float4 v[LB_WIN];
        const int n_local = sb->n_local;
        // Three tiles in flight: t0 (pass 2 this iteration), t1 (look-back
        // resolved this iteration, its records' loads issued last iteration),
        // t2 (pass 1 this iteration).  A tile's look-back therefore runs a full
        // iteration after every CTA published the aggregates it needs.
        ScanTile t0, t1, t2;
        auto start = [](ScanTile &T, int i, int B_, int L_) {
            T.tile = (int)blockIdx.x + i * (int)gridDim.x;
            T.b = T.tile % B_;
            T.c = T.tile / B_;
            T.Tc = min(T_TOK, L_ - T.c * T_TOK);
            T.r = i % REGIONS;
        };
        // pass 1 of local tile i (u landed, D1 ready)
        bool ok = true;
#define S5_FRONT(T, I)                                                                     \
    do {                                                                                   \
        if (wait_tile((I), sb, hdr) < 0) { ok = false; break; }                            \
        start((T), (I), B, L);                                                             \
        if (!pipe_wait(&sb->tmem_full[(T).r], ((I) / REGIONS) & 1, sb, hdr)) { ok = false; break; } \
        tc_fence_after();                                                                  \
        scan_front(cx, (T));                                                               \
    } while (0)
        if (n_local > 0) {
            S5_FRONT(t0, 0);
            if (ok && t0.pending) {
                scan_issue(cx, t0, v);
                scan_resolve(cx, t0, v);
            }
            if (ok && n_local > 1) {
                S5_FRONT(t1, 1);
                if (ok && t1.pending) scan_issue(cx, t1, v);
            }
        }
        for (int i = 0; ok && i < n_local; ++i) {
            if (i + 2 < n_local) {
                S5_FRONT(t2, i + 2);
                if (!ok) break;
            }
            if (i + 1 < n_local && t1.pending) scan_resolve(cx, t1, v);
            // pass 2 of tile i
            if (i >= 1 && !pipe_wait(&sb->xfree, (i - 1) & 1, sb, hdr)) break;
            const uint32_t col0 = lane_base + (uint32_t)t0.r * 128u;
            const float2 xend = (t0.Tc == T_TOK) ? pass2_full(col0, xb, kc, t0.carry, t0.elo)
                                                 : pass2_short(col0, xb, kc.lb, t0.carry, t0.Tc);
            if (t0.c == args.nchunks - 1 && args.x_last) args.x_last[(size_t)t0.b * P_M + m] = xend;
            fence_proxy_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&sb->xready);
            if (i + 2 < n_local && t2.pending) scan_issue(cx, t2, v);
            t0 = t1;
            t1 = t2;
        }
#undef S5_FRONT
    } else if (warp >= W_EPI && warp < W_EPI + 4) {
        // ------------------------------------------------------------ epilogue
        const int qd = warp - W_EPI;
        const int h = 32 * qd + lane;
        const float dh = args.d[h];
        const uint32_t lane_base = tmem + ((uint32_t)(32 * qd) << 16);
        const uint32_t hkb = (uint32_t)h >> 6, hc = (uint32_t)h & 63u;
        // offset inside a stage of (row q, this feature) in swizzle phase q;
        // row t lives at ub[t & 7] + (t >> 3) * 1024
        uint32_t ub[8];
#pragma unroll
        for (int q = 0; q < 8; ++q)
            ub[q] = hkb * (T_TOK * 128) + 128u * q + (((hc >> 3) ^ (uint32_t)q) << 4) + ((hc & 7u) << 1);
        const uint32_t stage0 = smem_addr(smem + SM_U);
        __nv_bfloat16 *yout = static_cast<__nv_bfloat16 *>(args.y);
        for (int i = 0;; ++i) {
            const int tile = wait_tile(i, sb, hdr);
            if (tile < 0) break;
            const int s = i % STAGES, r = i % REGIONS;
            const int b = tile % B, c = tile / B;
            const int Tc = min(T_TOK, L - c * T_TOK);
            if (!pipe_wait(&sb->mma2_done[r], (i / REGIONS) & 1, sb, hdr)) break;
            tc_fence_after();
            const uint32_t sbase = stage0 + (uint32_t)s * U_STAGE;
            __nv_bfloat16 *yrow = yout + ((size_t)b * L + (size_t)c * T_TOK) * H_F + h;
#pragma unroll
            for (int ch = 0; ch < T_TOK / 16; ++ch) {
                uint32_t yv[16];
                tmem_ld16(lane_base + (uint32_t)r * 128u + ch * 16, yv);
                tmem_wait_ld();
                if (ch == 3) {
                    // every column of the region has been read: it may be reused
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&sb->tmem_empty[r]);
                }
                float uf[16];
#pragma unroll
                for (int k = 0; k < 16; ++k) {
                    const int t = ch * 16 + k;
                    uf[k] = __uint_as_float(lds16(sbase + ub[t & 7] + (uint32_t)(t >> 3) * 1024u) << 16);
                }
                if (Tc == T_TOK) {
#pragma unroll
                    for (int k = 0; k < 16; ++k)
                        yrow[(size_t)(ch * 16 + k) * H_F] =
                            __float2bfloat16_rn(fmaf(dh, uf[k], __uint_as_float(yv[k])));
                } else {
#pragma unroll
                    for (int k = 0; k < 16; ++k)
                        if (ch * 16 + k < Tc)
                            yrow[(size_t)(ch * 16 + k) * H_F] =
                                __float2bfloat16_rn(fmaf(dh, uf[k], __uint_as_float(yv[k])));
                }
            }
            // u has been read: the stage may be refilled
            __syncwarp();
            if (lane == 0) mbar_arrive(&sb->empty_u[s]);
        }
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
// rows past L read as zero.
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

cudaError_t launch_forward_tc(const TcArgs &a, const void *u, cudaStream_t st, int num_sms) {
    CUtensorMap mu;
    if (!make_map(&mu, u, a.B, a.L)) return cudaErrorInvalidValue;
    const int words = P_M * H_F / 2 + H_F * P_M;
    weight_images_kernel<<<(words + 255) / 256, 256, 0, st>>>(a.b_bar, a.c_tilde, a.ws.wimg);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(fwd_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)SMEM_REQUEST);
    if (e != cudaSuccess) return e;
    // Cooperative launch: one CTA per SM, all resident, so the static wave
    // assignment never waits on a CTA that has not started.
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fwd_tc_kernel, THREADS, SMEM_REQUEST);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) return cudaErrorCooperativeLaunchTooLarge;
    const int grid = num_sms < a.ntiles ? num_sms : a.ntiles;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(THREADS);
    cfg.dynamicSmemBytes = SMEM_REQUEST;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, fwd_tc_kernel, mu, a);
}

}  // namespace s5
