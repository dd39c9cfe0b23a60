// s5_forward_tc.cu -- fused S5 forward on the 5th-generation tensor cores.
//
// Layer (review "S5: Simplified State Space Layers for Sequence Modeling", rows
// 1, 3, 4; summary "SIMPLIFIED STATE SPACE LAYERS ...", App. A and App. H):
//   Bu_k = B_bar u_k,  x_k = lambda_bar * x_{k-1} + Bu_k,  y_k = 2 Re(C~ x_k) + D u_k.
//
// Work split.  A sequence of nchunks tiles (64 tokens each) is spread over W
// "lanes" (CTAs): lane p of sequence b takes chunks p, p+W, p+2W, ...  With
// Lam = lambda_bar^64 and E(q) the end state of chunk q from a zero start
// (published by q's lane after its first scan pass), the state entering chunk
// q+1 is S(q+1) = Lam S(q) + E(q).  One more CTA per sequence, the sequence's
// scanner, runs exactly that chunk-level recurrence (in registers, one thread
// per mode): it reads each E(q) once and publishes every S(q).  Each lane then
// reads one record per tile: its carry.  Grid: B*(W+1) CTAs (one per SM,
// cooperative launch so that all are resident); when fewer than three CTAs per
// sequence fit, W = 1 and each CTA takes whole sequences with the carry passed
// on in registers.
//
// Each CTA runs a warp-specialised pipeline over its tiles:
//   warps 0-3   TMA and tcgen05.mma issue (one thread each):
//                 TMA: u tile [64 tokens x 128 features] bf16 -> smem (4
//                 stages, freed as soon as GEMM1 has read it); bulk copy of
//                 the two weight images at start-up
//                 GEMM1  Bu^T[2P x 64] = Bs[2P x H] * u^T      (into TMEM)
//                 GEMM2  y^T [H  x 64] = C'[H x 2P] * X^T      (into TMEM)
//               Each GEMM is split over two threads (rows / k-steps), so that
//               four chains of dependent MMAs are in flight.  Warp 2 also
//               allocates TMEM (512 columns: 4 regions of 128).
//   warps 4-7   scan, thread = mode = TMEM lane, pass 1 two tiles ahead: pass 1
//               of tile i+2 (end state from zero, published as the tile's
//               aggregate record), then pass 2 of tile i from its carry (two
//               interleaved 32-step chains), written as bf16 into the GEMM2
//               operand X [64 x 2P]
//   warps 8-11  epilogue, thread = feature = TMEM lane of GEMM2:
//               y = D2 + D*u (u re-read through L2), bf16 stores
//   warps 12-15 carries, thread = mode: wait for the tile's carry record and
//               put it into a shared-memory slot (two slots), ahead of the scan.
// The scanner CTAs run none of this: threads 0..P-1 only.
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
constexpr int THREADS = 512;
constexpr int W_TMEM = 2, W_SCAN = 4, W_EPI = 8, W_FOLD = 12;
constexpr int W_MAX = 64;               // lanes per sequence at most
constexpr int RB = 18;                  // aggregate records loaded per round
constexpr uint32_t BAR_SCAN = 1;        // named barrier of the four scan warps

constexpr uint32_t BS_BYTES = 2 * 2 * P_M * 128;       // [2 kb][2P rows][128 B]
constexpr uint32_t CP_BYTES = 4 * H_F * 128;           // [4 kb][H rows][128 B]
constexpr uint32_t SM_BS = 0;
constexpr uint32_t SM_CP = SM_BS + BS_BYTES;
constexpr uint32_t SM_U = SM_CP + CP_BYTES;            // [stage][2 kb][64 rows][128 B]
constexpr uint32_t U_STAGE = 2 * T_TOK * 128;
constexpr uint32_t SM_X = SM_U + STAGES * U_STAGE;     // [4 kb][64 rows][128 B]
constexpr uint32_t SM_CARRY = SM_X + 4 * T_TOK * 128;  // [2 slots][P] float2
constexpr uint32_t SM_BAR = SM_CARRY + 2 * P_M * 8;
constexpr uint32_t SM_TOTAL = SM_BAR + 256;
// Dynamic shared memory is requested up to the per-block limit; the slack
// absorbs the rounding of its base up to 1024 bytes (checked at run time).
constexpr uint32_t SMEM_REQUEST = 227 * 1024;
static_assert(SM_TOTAL <= SMEM_REQUEST, "shared memory budget");
static_assert(BS_BYTES + CP_BYTES == 8 * P_M * H_F, "image size");

constexpr unsigned long long PIPE_WAIT_NS = 2000000000ull;   // 2 s per pipeline wait
constexpr unsigned long long DRAIN_WAIT_NS = 200000000ull;   // 0.2 s per teardown wait

struct Bars {
    uint64_t full_u[STAGES], empty_u[STAGES];
    uint64_t tmem_full[REGIONS], tmem_empty[REGIONS], mma2_done[REGIONS];
    uint64_t xready, xfree, weights, drain;
    uint64_t carry_full[2], carry_empty[2];
    unsigned long long limit_ns;   // aggregate-record wait limit
    uint32_t tmem_base;
    unsigned epoch, drop;
    int abort;
};
static_assert(sizeof(Bars) <= 256, "barrier block");

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

// Barrier of `threads` threads that also returns the AND of `v` over them, so
// that the warps taking part leave a loop together.
__device__ __forceinline__ bool named_bar_and(uint32_t id, uint32_t threads, bool v) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.and.pred q, %2, %3, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)v), "r"(id), "r"(threads)
        : "memory");
    return r != 0;
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

__device__ __forceinline__ void sts32(uint32_t addr, uint32_t v) {
    asm volatile("st.shared.b32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
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

// ---------------------------------------------------------------------------
// Aggregate records.  Tile (b, c) (index b * nchunks + c) publishes, per mode,
// one 16-byte word {E.re, E.im, 0, epoch << 2 | FLAG_AGG}, written and read
// whole with GPU-scope relaxed vector accesses: a reader that sees this
// launch's tag sees the value stored with it, so one load both checks and
// fetches a record (no separate flag, no fence, one memory round trip).
// ---------------------------------------------------------------------------
__device__ __forceinline__ float4 ld_record(const float4 *p) {
    float4 v;
    asm volatile("ld.relaxed.gpu.global.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "l"(p)
                 : "memory");
    return v;
}
__device__ __forceinline__ void st_record(float4 *p, float2 e, unsigned tag) {
    asm volatile("st.relaxed.gpu.global.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(p), "f"(e.x), "f"(e.y),
                 "f"(0.f), "f"(__uint_as_float(tag))
                 : "memory");
}

// Lane geometry: CTA k of G.  W > 1: CTAs k < B*W are lanes (b = k % B,
// p = k / B) with chunks p, p + W, ...; CTAs k >= B*W are the scanners of
// sequences k - B*W.  W == 1: sequences k, k + G, ..., every chunk.
struct Lane {
    int B, W, G, k, nchunks;
    __device__ __forceinline__ bool scanner() const { return W > 1 && k >= B * W; }
    __device__ __forceinline__ int count() const {
        if (W > 1) return scanner() ? 0 : (nchunks - k / B + W - 1) / W;
        return (k < B ? (B - k + G - 1) / G : 0) * nchunks;
    }
    __device__ __forceinline__ void tile(int i, int &b, int &c) const {
        if (W > 1) {
            b = k % B;
            c = k / B + i * W;
        } else {
            b = k + (i / nchunks) * G;
            c = i % nchunks;
        }
    }
};

// Waits (bounded) until the 16-byte record at p carries `tag`; returns its
// value.  A wait that runs out latches S5_ERR_TIMEOUT (once per thread) and
// returns zero, so that the launch still completes.
__device__ float2 wait_record(const float4 *p, unsigned tag, WsHeader *hdr, unsigned long long limit,
                              bool &gave_up, unsigned tile) {
    float4 v = ld_record(p);
    if (__float_as_uint(v.w) == tag) return make_float2(v.x, v.y);
    const unsigned long long t0 = global_ns();
    while (!gave_up) {
        __nanosleep(64);
        v = ld_record(p);
        if (__float_as_uint(v.w) == tag) return make_float2(v.x, v.y);
        if (global_ns() - t0 > limit) {
            latch_status(hdr, S5_ERR_TIMEOUT);
            atomicCAS(&hdr->timeout_tile, 0u, tile + 1u);
            gave_up = true;
        }
    }
    return make_float2(0.f, 0.f);
}

// The sequence scanner (thread = mode m): S(0) = x0, then for every chunk q
// in order, publish S(q) (tag_s) and advance S(q+1) = Lam S(q) + E(q).  The
// aggregates E(q) (tag_e) of a group of R consecutive chunks are loaded in one
// round; the published prefix is folded and its S values go out at once, and
// the rest of the group is re-read in one round (bounded) until complete.
// R <= W: a group then spans at most two waves, and a lane's aggregate of
// wave g needs only its carry of wave g-2, so no group waits on its own
// carries.
__device__ __noinline__ void scanner_loop(const float4 *agg, float4 *carry, size_t seq, int nchunks, int R,
                                          float2 S, float2 Lam, unsigned tag_e, unsigned tag_s, WsHeader *hdr,
                                          unsigned long long limit) {
    bool gave_up = false;
    for (int q0 = 0; q0 < nchunks; q0 += R) {
        const int nr = min(R, nchunks - q0);
        const float4 *rp = agg + (seq + q0) * P_M;
        st_record(carry + (seq + q0) * P_M, S, tag_s);
        float4 v[RB];
        int done = 0;   // records of the group folded so far
        unsigned long long t0 = 0;
        bool timing = false;
        for (;;) {
#pragma unroll
            for (int w = 0; w < RB; ++w)
                if (w >= done && w < nr) v[w] = ld_record(rp + (size_t)w * P_M);
            bool prefix = true;
#pragma unroll
            for (int w = 0; w < RB; ++w) {
                if (w >= done && w < nr && prefix) {
                    if (__float_as_uint(v[w].w) == tag_e || gave_up) {
                        const bool ok = __float_as_uint(v[w].w) == tag_e;
                        S = cfma(Lam, S, ok ? make_float2(v[w].x, v[w].y) : make_float2(0.f, 0.f));
                        if (w + 1 < nr) st_record(carry + (seq + q0 + w + 1) * P_M, S, tag_s);
                        done = w + 1;
                    } else {
                        prefix = false;
                    }
                }
            }
            if (done >= nr) break;
            if (!timing) {
                t0 = global_ns();
                timing = true;
            } else if (global_ns() - t0 > limit) {
                latch_status(hdr, S5_ERR_TIMEOUT);
                atomicCAS(&hdr->timeout_tile, 0u, (unsigned)(seq + q0 + done) + 1u);
                gave_up = true;
            }
            __nanosleep(32);
        }
    }
}

// ---------------------------------------------------------------------------
// Scan passes over one tile of this thread's mode (TMEM lane): D1 columns
// [col0, col0+64) hold Re(Bu_t), [col0+64, col0+128) hold Im(Bu_t).
// ---------------------------------------------------------------------------
struct ScanConsts {
    float2 lb, lb32, lb64;   // lambda_bar and its powers
};

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
        tmem_ld16(col0 + ch * 16, re);
        tmem_ld16(col0 + 64 + ch * 16, im);
        tmem_wait_ld();
        const int n = Tc - ch * 16;
#pragma unroll
        for (int t = 0; t < 16; ++t)
            if (t < n) e = cfma(lb, e, make_float2(__uint_as_float(re[t]), __uint_as_float(im[t])));
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
            tmem_ld16(col0 + ch * 16, re);
            tmem_ld16(col0 + 64 + ch * 16, im);
            tmem_wait_ld();
        }
#pragma unroll
        for (int t = 0; t < 16; ++t) {
            uint32_t pv = 0;
            if (live && ch * 16 + t < Tc) {
                x = cfma(lb, x, make_float2(__uint_as_float(re[t]), __uint_as_float(im[t])));
                pv = pack_bf16(x.x, x.y);
            }
            sts32(xb[t & 7] + (uint32_t)((ch * 16 + t) >> 3) * 1024u, pv);
        }
    }
    return x;
}

// One tile in flight in the scan warps.
struct ScanTile {
    int g, b, c, Tc, r;
    float2 elo;
};

// Pass 1 of local tile i: waits for its GEMM1, runs pass 1 and publishes the
// tile's aggregate record for this mode.  Returns false if the wait gave up.
__device__ __forceinline__ bool scan_front(ScanTile &T, int i, const Lane &ln, int L, uint32_t lane_base,
                                           const ScanConsts &kc, float4 *rec, int m, unsigned tag,
                                           unsigned drop, Bars *sb, WsHeader *hdr) {
    ln.tile(i, T.b, T.c);
    T.g = T.b * ln.nchunks + T.c;
    T.Tc = min(T_TOK, L - T.c * T_TOK);
    T.r = i % REGIONS;
    if (!pipe_wait(&sb->tmem_full[T.r], (i / REGIONS) & 1, sb, hdr)) return false;
    tc_fence_after();
    const uint32_t col0 = lane_base + (uint32_t)T.r * 128u;
    T.elo = make_float2(0.f, 0.f);
    const float2 E = (T.Tc == T_TOK) ? pass1_full(col0, kc, T.elo) : pass1_short(col0, T.Tc, kc.lb);
    if (drop != (unsigned)T.g + 1u) st_record(rec + (size_t)T.g * P_M + m, E, tag);
    return true;
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
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    const uint32_t pad = (1024u - (smem_addr(smem_raw) & 1023u)) & 1023u;
    unsigned char *smem = smem_raw + pad;
    Bars *sb = reinterpret_cast<Bars *>(smem + SM_BAR);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    WsHeader *hdr = args.ws.hdr;
    float4 *rec = args.ws.agg;         // [ntiles][P] aggregate records
    const int B = args.B, L = args.L, nchunks = args.nchunks, W = args.W;
    Lane ln;
    ln.B = B;
    ln.W = W;
    ln.G = (int)gridDim.x;
    ln.k = (int)blockIdx.x;
    ln.nchunks = nchunks;
    const int n = ln.count();
    const bool scanner = ln.scanner();
    // the allocation must hold the 1024-aligned layout (the same for every thread)
    const bool fits = pad + SM_TOTAL <= SMEM_REQUEST;

    if (fits && scanner) {
        // ------------------------------------------------------------ sequence scanner
        if (threadIdx.x < P_M) {
            const int m = threadIdx.x, b = ln.k - B * W;
            const unsigned ep = *reinterpret_cast<volatile unsigned *>(&hdr->epoch);
            const unsigned lim = *reinterpret_cast<volatile unsigned *>(&hdr->wait_limit_us);
            const float2 S0 = args.x0 ? args.x0[(size_t)b * P_M + m] : make_float2(0.f, 0.f);
            scanner_loop(args.ws.agg + m, args.ws.carry + m, (size_t)b * nchunks, nchunks, min(RB, W), S0,
                         cpow(args.lambda_bar[m], 64), (ep << 2) | FLAG_AGG, (ep << 2) | FLAG_INCL, hdr,
                         1000ull * (lim ? lim : 1000000u));
        }
    } else if (fits) {
        if (threadIdx.x == 0) {
            for (int s = 0; s < STAGES; ++s) {
                mbar_init(&sb->full_u[s], 1);
                mbar_init(&sb->empty_u[s], 2);   // the two GEMM1 halves
            }
            for (int r = 0; r < REGIONS; ++r) {
                mbar_init(&sb->tmem_full[r], 2);   // the two GEMM1 halves
                mbar_init(&sb->tmem_empty[r], 4);  // the four epilogue warps
                mbar_init(&sb->mma2_done[r], 2);   // the two GEMM2 halves
            }
            mbar_init(&sb->xready, 4);
            mbar_init(&sb->xfree, 2);
            mbar_init(&sb->weights, 1);
            mbar_init(&sb->drain, 4);          // the four issuing threads
            for (int q = 0; q < 2; ++q) {
                mbar_init(&sb->carry_full[q], 4);    // the four fold warps
                mbar_init(&sb->carry_empty[q], 4);   // the four scan warps
            }
            sb->abort = 0;
            fence_mbar_init();
            sb->epoch = *reinterpret_cast<volatile unsigned *>(&hdr->epoch);
            sb->drop = *reinterpret_cast<volatile unsigned *>(&hdr->drop_publish);
            const unsigned lim = *reinterpret_cast<volatile unsigned *>(&hdr->wait_limit_us);
            sb->limit_ns = 1000ull * (lim ? lim : 1000000u);
        }
        if (warp == W_TMEM) {
            tmem_alloc(&sb->tmem_base, 512);
            tmem_relinquish();
        }
    } else if (threadIdx.x == 0) {
        latch_status(hdr, S5_ERR_UNSUPPORTED);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const bool pipeline = fits && !scanner;
    const uint32_t tmem = pipeline ? sb->tmem_base : 0u;
    const unsigned tag = pipeline ? ((sb->epoch << 2) | FLAG_AGG) : 0u;

    if (!pipeline) {
        // nothing to run: straight to the teardown
    } else if (warp < 4) {
        // ------------------------------------------------------------ TMA + MMA issue
        // One dependent chain of 8 MMAs per thread and tile: a single thread
        // issues a chain of accumulating MMAs at roughly one per 235 cycles, so
        // the tile's 32 MMAs are spread over four issuing threads.
        //   warp 1: GEMM1 rows 0..P-1 (Re),  warp 2: GEMM1 rows P..2P-1 (Im),
        //   warp 3: GEMM2 k-steps 0..7,      warp 0: GEMM2 k-steps 8..15 and the
        //   TMA producer.  GEMM2's two halves accumulate into columns 0..63 and
        //   64..127 of the tile's region; the epilogue adds them.
        if (lane == 0) {
            const uint32_t idesc = idesc_bf16_f32(128, T_TOK);
            const uint32_t bs = smem_addr(smem + SM_BS), cp = smem_addr(smem + SM_CP);
            const uint32_t xs = smem_addr(smem + SM_X);
            if (warp == 0) {
                prefetch_tmap(&tmap_u);
                mbar_arrive_tx(&sb->weights, BS_BYTES + CP_BYTES);
                bulk_load(smem + SM_BS, args.ws.wimg + SM_BS, BS_BYTES, &sb->weights);
                bulk_load(smem + SM_CP, args.ws.wimg + SM_CP, CP_BYTES, &sb->weights);
            }
            bool ok = n == 0 || pipe_wait(&sb->weights, 0, sb, hdr);
            if (warp == 1 || warp == 2) {
                const int mb = warp - 1;
                for (int g = 0; ok && g < n; ++g) {
                    const int s = g % STAGES, r = g % REGIONS;
                    ok = pipe_wait(&sb->full_u[s], (g / STAGES) & 1, sb, hdr) &&
                         (g < REGIONS || pipe_wait(&sb->tmem_empty[r], ((g / REGIONS) - 1) & 1, sb, hdr));
                    if (!ok) break;
                    tc_fence_after();
                    const uint32_t ub = smem_addr(smem + SM_U + s * U_STAGE);
#pragma unroll
                    for (int kq = 0; kq < H_F / 16; ++kq)
                        mma_bf16(tmem + (uint32_t)r * 128u + (uint32_t)mb * 64u,
                                 sw128_kmajor_desc(bs + (kq >> 2) * (2 * P_M * 128) + mb * (P_M * 128) + (kq & 3) * 32),
                                 sw128_kmajor_desc(ub + (kq >> 2) * (T_TOK * 128) + (kq & 3) * 32), idesc, kq > 0);
                    mma_commit(&sb->tmem_full[r]);
                    mma_commit(&sb->empty_u[s]);
                }
            } else {
                // GEMM2 half hf (and, in warp 0, the u loads)
                const int hf = warp == 3 ? 0 : 1;
                int g2 = 0, il = 0;   // next tile for GEMM2 / for a u load
                int last_issue[STAGES];
                for (int q = 0; q < STAGES; ++q) last_issue[q] = -1;
                const int nl = warp == 0 ? n : 0;
                unsigned long long t0 = global_ns();
                while (ok && (g2 < n || il < nl)) {
                    bool progress = false;
                    if (il < nl) {
                        const int s = il % STAGES;
                        if (il < STAGES || mbar_test_wait(&sb->empty_u[s], ((il / STAGES) - 1) & 1)) {
                            int b, c;
                            ln.tile(il, b, c);
                            unsigned char *dst = smem + SM_U + s * U_STAGE;
                            mbar_arrive_tx(&sb->full_u[s], U_STAGE);
                            tma_load_3d(dst, &tmap_u, 0, c * T_TOK, b, &sb->full_u[s]);
                            tma_load_3d(dst + T_TOK * 128, &tmap_u, 64, c * T_TOK, b, &sb->full_u[s]);
                            last_issue[s] = il;
                            ++il;
                            progress = true;
                        }
                    }
                    if (g2 < n && mbar_test_wait(&sb->xready, g2 & 1)) {
                        tc_fence_after();
                        const uint32_t d = tmem + (uint32_t)(g2 % REGIONS) * 128u + (uint32_t)hf * 64u;
#pragma unroll
                        for (int k8 = 0; k8 < 8; ++k8) {
                            const int kq = hf * 8 + k8;
                            mma_bf16(d, sw128_kmajor_desc(cp + (kq >> 2) * (H_F * 128) + (kq & 3) * 32),
                                     sw128_kmajor_desc(xs + (kq >> 2) * (T_TOK * 128) + (kq & 3) * 32), idesc,
                                     k8 > 0);
                        }
                        mma_commit(&sb->mma2_done[g2 % REGIONS]);
                        mma_commit(&sb->xfree);
                        ++g2;
                        progress = true;
                    }
                    if (progress) {
                        t0 = global_ns();
                    } else if (aborted(sb)) {
                        break;
                    } else if (global_ns() - t0 > PIPE_WAIT_NS) {
                        set_abort(sb, hdr);
                        break;
                    } else {
                        __nanosleep(32);
                    }
                }
                if (warp == 0) {
                    // copies still in flight must land before the CTA exits
                    drain_wait(&sb->weights, 0);
                    for (int q = 0; q < STAGES; ++q)
                        if (last_issue[q] >= 0) drain_wait(&sb->full_u[q], (last_issue[q] / STAGES) & 1);
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
        kc.lb32 = cpow(kc.lb, 32);
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
        const float2 *slots = reinterpret_cast<const float2 *>(smem + SM_CARRY);
        const unsigned drop = sb->drop;

        // Every exit from this loop is decided by named_bar_and, so the four
        // warps always meet at the same barriers.
        ScanTile t0, t1, t2;
        bool alive = true;
        for (int j = 0; j < 2 && j < n; ++j) {
            ScanTile &T = j == 0 ? t0 : t1;
            const bool mine = scan_front(T, j, ln, L, lane_base, kc, rec, m, tag, drop, sb, hdr);
            if (!named_bar_and(BAR_SCAN, 128, mine)) {
                alive = false;
                break;
            }
        }
        float2 xprev = make_float2(0.f, 0.f);
        bool mine = true;
        for (int i = 0; alive && i < n; ++i) {
            const bool front = i + 2 < n;
            if (mine && front)
                mine = scan_front(t2, i + 2, ln, L, lane_base, kc, rec, m, tag, drop, sb, hdr);
            if (!named_bar_and(BAR_SCAN, 128, mine)) break;
            // carry of tile i: from the carry warps' slot, or (one lane per
            // sequence) the previous tile's end state
            float2 carry = xprev;
            if (W > 1) {
                mine = pipe_wait(&sb->carry_full[i & 1], (i >> 1) & 1, sb, hdr);
                if (mine) {
                    carry = slots[(i & 1) * P_M + m];
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&sb->carry_empty[i & 1]);
                }
            } else if (t0.c == 0) {
                carry = args.x0 ? args.x0[(size_t)t0.b * P_M + m] : make_float2(0.f, 0.f);
            }
            if (mine) {
                // pass 2 of tile i once GEMM2 of tile i-1 has read X
                mine = i == 0 || pipe_wait(&sb->xfree, (i - 1) & 1, sb, hdr);
                if (mine) {
                    tc_fence_after();
                    const uint32_t col0 = lane_base + (uint32_t)t0.r * 128u;
                    xprev = (t0.Tc == T_TOK) ? pass2_full(col0, xb, kc, carry, t0.elo)
                                             : pass2_short(col0, xb, kc.lb, carry, t0.Tc);
                    if (t0.c == nchunks - 1 && args.x_last) args.x_last[(size_t)t0.b * P_M + m] = xprev;
                    fence_proxy_async_smem();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&sb->xready);
                }
            }
            t0 = t1;
            t1 = t2;
        }
    } else if (warp >= W_EPI && warp < W_EPI + 4) {
        // ------------------------------------------------------------ epilogue
        const int qd = warp - W_EPI;
        const int h = 32 * qd + lane;
        const float dh = args.d[h];
        const uint32_t lane_base = tmem + ((uint32_t)(32 * qd) << 16);
        const __nv_bfloat16 *uin = static_cast<const __nv_bfloat16 *>(args.u);
        __nv_bfloat16 *yout = static_cast<__nv_bfloat16 *>(args.y);
        for (int i = 0; i < n; ++i) {
            const int r = i % REGIONS;
            int b, c;
            ln.tile(i, b, c);
            const int Tc = min(T_TOK, L - c * T_TOK);
            const size_t row0 = ((size_t)b * L + (size_t)c * T_TOK) * H_F + h;
            // this feature's u over the tile, loaded before the wait so that
            // the latency overlaps it
            __nv_bfloat16 uv[T_TOK];
#pragma unroll
            for (int k = 0; k < T_TOK; ++k)
                uv[k] = (k < Tc) ? uin[row0 + (size_t)k * H_F] : __float2bfloat16_rn(0.f);
            if (!pipe_wait(&sb->mma2_done[r], (i / REGIONS) & 1, sb, hdr)) break;
            tc_fence_after();
            __nv_bfloat16 *yrow = yout + row0;
#pragma unroll
            for (int ch = 0; ch < T_TOK / 16; ++ch) {
                uint32_t ya[16], yb[16];
                tmem_ld16(lane_base + (uint32_t)r * 128u + ch * 16, ya);
                tmem_ld16(lane_base + (uint32_t)r * 128u + 64u + ch * 16, yb);
                tmem_wait_ld();
                float yv[16];
#pragma unroll
                for (int k = 0; k < 16; ++k) yv[k] = __uint_as_float(ya[k]) + __uint_as_float(yb[k]);
                if (ch == 3) {
                    // every column of the region has been read: it may be reused
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&sb->tmem_empty[r]);
                }
#pragma unroll
                for (int k = 0; k < 16; ++k)
                    if (ch * 16 + k < Tc)
                        yrow[(size_t)(ch * 16 + k) * H_F] =
                            __float2bfloat16_rn(fmaf(dh, __bfloat162float(uv[ch * 16 + k]), yv[k]));
            }
        }
    } else if (warp >= W_FOLD && warp < W_FOLD + 4 && W > 1) {
        // ------------------------------------------------------------ carries
        const int m = 32 * (warp - W_FOLD) + lane;
        float2 *slots = reinterpret_cast<float2 *>(smem + SM_CARRY);
        const float4 *carry = args.ws.carry;
        const unsigned tag_s = (sb->epoch << 2) | FLAG_INCL;
        const unsigned long long limit = sb->limit_ns;
        const int b = ln.k % B, p = ln.k / B;
        const size_t seq = (size_t)b * nchunks;
        bool gave_up = false;
        for (int j = 0; j < n; ++j) {
            // slot j % 2 is free once the scan has read tile j-2's carry
            if (j >= 2 && !pipe_wait(&sb->carry_empty[j & 1], ((j >> 1) - 1) & 1, sb, hdr)) break;
            const float2 own = wait_record(carry + (seq + (size_t)j * W + p) * P_M + m, tag_s, hdr, limit,
                                           gave_up, (unsigned)(seq + (size_t)j * W + p));
            slots[(j & 1) * P_M + m] = own;
            __syncwarp();
            if (lane == 0) mbar_arrive(&sb->carry_full[j & 1]);
        }
    }

    // ---------------------------------------------------------------- teardown
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (pipeline && warp == W_TMEM) tmem_dealloc(tmem, 512);
    if (threadIdx.x == 0) {
        __threadfence();
        const unsigned prev = atomicAdd(&hdr->done_counter, 1u);
        if (prev == gridDim.x - 1) {
            const unsigned e = *reinterpret_cast<volatile unsigned *>(&hdr->epoch);
            hdr->tile_counter = 0;
            hdr->done_counter = 0;
            hdr->epoch = (e + 1) & 0x3FFFFFFFu;
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

// Lanes per sequence and grid: W lanes plus one scanner per sequence, B*(W+1)
// CTAs (2 <= W <= nchunks, W <= W_MAX), when at least three CTAs per sequence
// fit on the SMs; else W = 1, min(B, SMs) CTAs, each taking whole sequences.
void tc_grid(int B, int nchunks, int num_sms, int *W, int *G) {
    int w = B <= num_sms ? num_sms / B - 1 : 0;
    if (w > nchunks) w = nchunks;
    if (w > W_MAX) w = W_MAX;
    if (w >= 2) {
        *W = w;
        *G = B * (w + 1);
    } else {
        *W = 1;
        *G = B < num_sms ? B : num_sms;
    }
}

cudaError_t launch_forward_tc(const TcArgs &a0, const void *u, cudaStream_t st, int num_sms) {
    TcArgs a = a0;
    a.u = u;
    int G = 0;
    tc_grid(a.B, a.nchunks, num_sms, &a.W, &G);
    CUtensorMap mu;
    if (!make_map(&mu, u, a.B, a.L)) return cudaErrorInvalidValue;
    const int words = P_M * H_F / 2 + H_F * P_M;
    weight_images_kernel<<<(words + 255) / 256, 256, 0, st>>>(a.b_bar, a.c_tilde, a.ws.wimg);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(fwd_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)SMEM_REQUEST);
    if (e != cudaSuccess) return e;
    // Cooperative launch: one CTA per SM, all resident, so a lane never waits
    // on a CTA that has not started.
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fwd_tc_kernel, THREADS, SMEM_REQUEST);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) return cudaErrorCooperativeLaunchTooLarge;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)G);
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
