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
//   warp 0      TMA: u tile [64 tokens x 128 features] bf16 -> smem (3 stages,
//               freed once GEMM1 has read it); bulk copy of the two weight
//               images at start-up
//   warp 1      GEMM1  Bu^T[2P x 64] = Bs[2P x H] * u^T  (16 MMAs from one
//               thread into the tile's TMEM region: Re rows, then Im rows)
//   warp 2      GEMM2  y^T [H  x 64] = C'[H x 2P] * X^T  (16 MMAs from one
//               thread into columns 0..63 of the region, once X is complete);
//               TMEM allocation (512 columns: 4 regions of 128)
//   warp 3      a second TMA copy of each tile's u, for the epilogue
//   warps 4-7   scan, thread = mode = TMEM lane, pass 1 two tiles ahead: pass 1
//               of tile i+2 (four 16-token chains from zero; the tile's end
//               state is published as its aggregate record), then pass 2 of
//               tile i (the four chains from the carry), written as bf16 into
//               the GEMM2 operand X [64 x 2P]
//   warps 8-11  epilogue, thread = feature = TMEM lane of GEMM2:
//               y = acc + D*u (u from the shared copy), bf16 stores
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
// Compiled twice.  S5_TC_REV = 0 (this file): the layer's forward scan.
// S5_TC_REV = 1 (s5_backward_tc.cu includes this file): the backward scan of
// the bidirectional layer -- chunks and the tokens inside a tile are visited
// in reverse (scan position q is chunk nchunks-1-q, token 63-s of a full
// tile), x0 and x_last are not used, and the epilogue adds the readout to the
// y already there: its second TMA copy reads y instead of u.  Every
// difference sits in an "#if S5_TC_REV" block.
#ifndef S5_TC_REV
#define S5_TC_REV 0
#endif
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
constexpr int W_TMEM = 2, W_SCAN = 4, W_EPI = 8, W_FOLD = 12;
constexpr int W_MAX = 64;               // lanes per sequence at most
constexpr int TC_FREE_SMS = 8;          // SMs left to the next kernel (see tc_grid)
constexpr int RB = 18;                  // aggregate records loaded per round

constexpr uint32_t BS_BYTES = 2 * 2 * P_M * 128;       // [2 kb][2P rows][128 B]
constexpr uint32_t CP_BYTES = 4 * H_F * 128;           // [4 kb][H rows][128 B]
constexpr uint32_t SM_BS = 0;
constexpr uint32_t SM_CP = SM_BS + BS_BYTES;
constexpr uint32_t SM_U = SM_CP + CP_BYTES;            // [stage][2 kb][64 rows][128 B]
constexpr uint32_t U_STAGE = 2 * T_TOK * 128;
constexpr uint32_t SM_EU = SM_U + STAGES * U_STAGE;    // the epilogue's copy of u: [2 kb][64 rows][128 B]
constexpr uint32_t SM_X = SM_EU + U_STAGE;             // [4 kb][64 rows][128 B]
constexpr uint32_t SM_CARRY = SM_X + 4 * T_TOK * 128;  // [2 slots][P] float2
constexpr uint32_t SM_BAR = SM_CARRY + 2 * P_M * 8;
constexpr uint32_t SM_TOTAL = SM_BAR + 512;
// Dynamic shared memory is requested up to the per-block limit; the slack
// absorbs the rounding of its base up to 1024 bytes (checked at run time).
constexpr uint32_t SMEM_REQUEST = 227 * 1024;
static_assert(SM_TOTAL <= SMEM_REQUEST, "shared memory budget");
static_assert(BS_BYTES + CP_BYTES == 8 * P_M * H_F, "image size");

constexpr unsigned long long PIPE_WAIT_NS = 2000000000ull;   // 2 s per pipeline wait
constexpr unsigned long long DRAIN_WAIT_NS = 200000000ull;   // 0.2 s per teardown wait

struct Bars {
    uint64_t full_u[STAGES], empty_u[STAGES];
    uint64_t eu_full, eu_empty;     // the epilogue's u buffer
    uint64_t tmem_full[REGIONS], tmem_empty[REGIONS], mma2_done[REGIONS];
    uint64_t xready, xfree;         // X written by the four scan warps / read by GEMM2
    uint64_t weights, drain;
    uint64_t carry_full[2], carry_empty[2];
    unsigned long long limit_ns;   // aggregate-record wait limit
    uint32_t tmem_base;
    unsigned epoch, drop;
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
__device__ __forceinline__ bool pipe_wait_slow(uint64_t *bar, uint32_t parity, Bars *sb, WsHeader *hdr) {
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
__device__ __forceinline__ bool pipe_wait(uint64_t *bar, uint32_t parity, Bars *sb, WsHeader *hdr) {
    return mbar_try_wait(bar, parity) || pipe_wait_slow(bar, parity, sb, hdr);
}
// Teardown wait: bounded, ignores the abort flag.
__device__ __forceinline__ bool drain_wait(uint64_t *bar, uint32_t parity) {
    const unsigned long long t0 = global_ns();
    while (!mbar_try_wait_sleep(bar, parity, SLEEP_HINT_NS))
        if (global_ns() - t0 > DRAIN_WAIT_NS) return false;
    return true;
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
    int kb, kp;   // k % B and k / B, computed once
    __device__ __forceinline__ void init() {
        kb = k % B;
        kp = k / B;
    }
    __device__ __forceinline__ bool scanner() const { return W > 1 && k >= B * W; }
    __device__ __forceinline__ int count() const {
        if (W > 1) return scanner() ? 0 : (nchunks - kp + W - 1) / W;
        return (k < B ? (B - k + G - 1) / G : 0) * nchunks;
    }
    __device__ __forceinline__ void tile(int i, int &b, int &c) const {
        if (W > 1) {
            b = kb;
            c = kp + i * W;
        } else {
            b = k + (i / nchunks) * G;
            c = i % nchunks;
        }
    }
};

// Waits (bounded) until the 16-byte record at p carries `tag`; returns its
// value.  The record is re-read back to back (each read is one L2 round
// trip): a sleep between reads measurably delays the carries.  A wait that runs out latches S5_ERR_TIMEOUT (once per thread) and
// returns zero, so that the launch still completes.
__device__ float2 wait_record(const float4 *p, unsigned tag, WsHeader *hdr, unsigned long long limit,
                              bool &gave_up, unsigned tile) {
    float4 v = ld_record(p);
    if (__float_as_uint(v.w) == tag) return make_float2(v.x, v.y);
    const unsigned long long t0 = global_ns();
    while (!gave_up) {
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
        }
    }
}

// ---------------------------------------------------------------------------
// Scan passes over one tile of this thread's mode (TMEM lane): columns
// [col0, col0+64) hold Re(Bu_t), [col0+64, col0+128) hold Im(Bu_t).  A full
// tile runs as four independent 16-token chains (tokens 16q .. 16q+15), so
// that the FMA pipe, not the chain's latency, sets the pace.
// ---------------------------------------------------------------------------
struct ScanConsts {
    float2 lb, lb16;   // lambda_bar, lambda_bar^16
};

// Full tile, pass 1: the four chains' end states from zero (e[0..2] kept for
// pass 2); returns the tile's end state from zero, (((e0 L + e1) L + e2) L + e3)
// with L = lambda_bar^16.
__device__ __forceinline__ float2 pass1_full(uint32_t col0, const ScanConsts &k, float2 (&e)[3]) {
    float2 c0 = make_float2(0.f, 0.f), c1 = c0, c2 = c0, c3 = c0;
#pragma unroll 1
    for (int r = 0; r < 4; ++r) {
        uint32_t re[4][4], im[4][4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
#if S5_TC_REV
            tmem_ld4(col0 + 60 - 16 * q - 4 * r, re[q]);
            tmem_ld4(col0 + 64 + 60 - 16 * q - 4 * r, im[q]);
#else
            tmem_ld4(col0 + 16 * q + 4 * r, re[q]);
            tmem_ld4(col0 + 64 + 16 * q + 4 * r, im[q]);
#endif
        }
        tmem_wait_ld();
#pragma unroll
#if S5_TC_REV
        for (int tt = 0; tt < 4; ++tt) {
            const int t = 3 - tt;
#else
        for (int t = 0; t < 4; ++t) {
#endif
            c0 = cfma(k.lb, c0, make_float2(__uint_as_float(re[0][t]), __uint_as_float(im[0][t])));
            c1 = cfma(k.lb, c1, make_float2(__uint_as_float(re[1][t]), __uint_as_float(im[1][t])));
            c2 = cfma(k.lb, c2, make_float2(__uint_as_float(re[2][t]), __uint_as_float(im[2][t])));
            c3 = cfma(k.lb, c3, make_float2(__uint_as_float(re[3][t]), __uint_as_float(im[3][t])));
        }
    }
    e[0] = c0;
    e[1] = c1;
    e[2] = c2;
    return cfma(k.lb16, cfma(k.lb16, cfma(k.lb16, c0, c1), c2), c3);
}

// Short tile (Tc < 64): end state from zero over its Tc tokens.
__device__ __noinline__ float2 pass1_short(uint32_t col0, int Tc, float2 lb) {
    float2 e = make_float2(0.f, 0.f);
#pragma unroll 1
#if S5_TC_REV
    for (int ch = (Tc - 1) / 16; ch >= 0; --ch) {
#else
    for (int ch = 0; ch * 16 < Tc; ++ch) {
#endif
        uint32_t re[16], im[16];
        tmem_ld16(col0 + ch * 16, re);
        tmem_ld16(col0 + 64 + ch * 16, im);
        tmem_wait_ld();
        const int n = Tc - ch * 16;
#pragma unroll
#if S5_TC_REV
        for (int t = 15; t >= 0; --t)
#else
        for (int t = 0; t < 16; ++t)
#endif
            if (t < n) e = cfma(lb, e, make_float2(__uint_as_float(re[t]), __uint_as_float(im[t])));
    }
    return e;
}

// Full tile, pass 2: the four chains start from the carry S and
// S_{q+1} = L S_q + e_q; every state goes as bf16 (Re, Im) into row t of X
// (row t at xb[t & 7] + (t >> 3) * 1024).  `done` is arrived once the last
// Bu column is in registers.  Returns the state after token 63.
__device__ __forceinline__ float2 pass2_full(uint32_t col0, const uint32_t (&xb)[8], const ScanConsts &k,
                                             float2 S, const float2 (&e)[3]) {
    float2 s0 = S;
    float2 s1 = cfma(k.lb16, s0, e[0]);
    float2 s2 = cfma(k.lb16, s1, e[1]);
    float2 s3 = cfma(k.lb16, s2, e[2]);
    // rounds of 4 tokens per chain (token 16q + 4r + t is row (2q + r/2) * 8 + (r%2)*4 + t)
#pragma unroll 1
    for (int r = 0; r < 4; ++r) {
        uint32_t re[4][4], im[4][4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
#if S5_TC_REV
            tmem_ld4(col0 + 60 - 16 * q - 4 * r, re[q]);
            tmem_ld4(col0 + 64 + 60 - 16 * q - 4 * r, im[q]);
#else
            tmem_ld4(col0 + 16 * q + 4 * r, re[q]);
            tmem_ld4(col0 + 64 + 16 * q + 4 * r, im[q]);
#endif
        }
        tmem_wait_ld();
        const uint32_t o = (uint32_t)(r >> 1) * 1024u;
        const int t0 = (r & 1) * 4;
#pragma unroll
#if S5_TC_REV
        // scan position 16q + 4r + tt is token and X row 63 - (16q + 4r + tt)
        for (int tt = 0; tt < 4; ++tt) {
            const int t = 3 - tt;
#else
        for (int t = 0; t < 4; ++t) {
#endif
            s0 = cfma(k.lb, s0, make_float2(__uint_as_float(re[0][t]), __uint_as_float(im[0][t])));
            s1 = cfma(k.lb, s1, make_float2(__uint_as_float(re[1][t]), __uint_as_float(im[1][t])));
            s2 = cfma(k.lb, s2, make_float2(__uint_as_float(re[2][t]), __uint_as_float(im[2][t])));
            s3 = cfma(k.lb, s3, make_float2(__uint_as_float(re[3][t]), __uint_as_float(im[3][t])));
#if S5_TC_REV
            const uint32_t a = ((r & 1) ? xb[3 - tt] : xb[7 - tt]) + 7168u - o;
            sts32(a, pack_bf16(s0.x, s0.y));
            sts32(a - 2048u, pack_bf16(s1.x, s1.y));
            sts32(a - 4096u, pack_bf16(s2.x, s2.y));
            sts32(a - 6144u, pack_bf16(s3.x, s3.y));
#else
            const uint32_t a = ((r & 1) ? xb[4 + t] : xb[t]) + o;
            sts32(a, pack_bf16(s0.x, s0.y));
            sts32(a + 2048u, pack_bf16(s1.x, s1.y));
            sts32(a + 4096u, pack_bf16(s2.x, s2.y));
            sts32(a + 6144u, pack_bf16(s3.x, s3.y));
#endif
        }
        (void)t0;
    }
    return s3;
}

// Short tile: sequential states; rows past Tc are written as zeros.
__device__ __noinline__ float2 pass2_short(uint32_t col0, const uint32_t (&xb)[8], float2 lb, float2 x, int Tc) {
#pragma unroll 1
#if S5_TC_REV
    for (int ch = T_TOK / 16 - 1; ch >= 0; --ch) {
#else
    for (int ch = 0; ch < T_TOK / 16; ++ch) {
#endif
        uint32_t re[16], im[16];
        const bool live = ch * 16 < Tc;
        if (live) {
            tmem_ld16(col0 + ch * 16, re);
            tmem_ld16(col0 + 64 + ch * 16, im);
            tmem_wait_ld();
        }
#pragma unroll
#if S5_TC_REV
        for (int t = 15; t >= 0; --t) {
#else
        for (int t = 0; t < 16; ++t) {
#endif
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

// One tile in flight in the scan warps: its length and pass-1 chain states.
struct ScanTile {
    int Tc;
    float2 e[3];
};

// Pass 1 of local tile i: waits for its GEMM1, runs pass 1 and publishes the
// tile's aggregate record for this mode.  Returns false if the wait gave up.
__device__ __forceinline__ bool scan_front(ScanTile &T, int i, const Lane &ln, int L, uint32_t lane_base,
                                           const ScanConsts &kc, float4 *rec, int m, unsigned tag,
                                           unsigned drop, Bars *sb, WsHeader *hdr) {
    int b, c;
    ln.tile(i, b, c);
    const int g = b * ln.nchunks + c, r = i % REGIONS;
#if S5_TC_REV
    T.Tc = min(T_TOK, L - (ln.nchunks - 1 - c) * T_TOK);
#else
    T.Tc = min(T_TOK, L - c * T_TOK);
#endif
    if (!pipe_wait(&sb->tmem_full[r], (i / REGIONS) & 1, sb, hdr)) return false;
    tc_fence_after();
    const uint32_t col0 = lane_base + (uint32_t)r * 128u;
    float2 E;
    if (T.Tc == T_TOK) {
        E = pass1_full(col0, kc, T.e);
    } else {
        E = pass1_short(col0, T.Tc, kc.lb);
        T.e[0] = T.e[1] = T.e[2] = make_float2(0.f, 0.f);
    }
    if (drop != (unsigned)g + 1u) st_record(rec + (size_t)g * P_M + m, E, tag);
    return true;
}

// ---------------------------------------------------------------------------
// Prep: bf16 operand images in the exact byte layout the MMA descriptors read.
// ---------------------------------------------------------------------------
__global__ void weight_images_kernel(const float2 *__restrict__ b_bar, const float2 *__restrict__ c_tilde,
                                     unsigned char *__restrict__ img) {
    // launched programmatically: the scan kernel after it may be scheduled
    // at once; B_bar and C~ are read, and the images written, only after the
    // previous kernel (which may produce the former or read the latter) ends
    griddep_launch_dependents();
    griddep_wait();
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
#if S5_TC_REV
bwd_tc_kernel(const __grid_constant__ CUtensorMap tmap_u, const __grid_constant__ CUtensorMap tmap_e,
              const TcArgs args) {
#else
fwd_tc_kernel(const __grid_constant__ CUtensorMap tmap_u, const TcArgs args) {
#endif
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    const uint32_t pad = (1024u - (smem_addr(smem_raw) & 1023u)) & 1023u;
    unsigned char *smem = smem_raw + pad;
    Bars *sb = reinterpret_cast<Bars *>(smem + SM_BAR);
    // A kernel launched programmatically after this one (the next layer's
    // discretisation, say) may be scheduled at once: its blocks take SMs as
    // this kernel's CTAs exit, and it waits for this grid before touching
    // anything this grid reads or writes.
    griddep_launch_dependents();

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
    ln.init();
    const int n = ln.count();
    const bool scanner = ln.scanner();
    // the allocation must hold the 1024-aligned layout (the same for every thread)
    const bool fits = pad + SM_TOTAL <= SMEM_REQUEST;

    if (fits && scanner) {
        // ------------------------------------------------------------ sequence scanner
        griddep_wait();
        if (threadIdx.x < P_M) {
            const int m = threadIdx.x, b = ln.k - B * W;
            // the header's words in two independent 16-byte loads (the
            // workspace is 16-byte aligned): epoch is word 3, the wait limit word 5
            const uint4 h0 = __ldcg(reinterpret_cast<const uint4 *>(hdr));
            const uint4 h1 = __ldcg(reinterpret_cast<const uint4 *>(hdr) + 1);
            const unsigned ep = h0.w, lim = h1.y;
            const float2 S0 = args.x0 ? args.x0[(size_t)b * P_M + m] : make_float2(0.f, 0.f);
            scanner_loop(args.ws.agg + m, args.ws.carry + m, (size_t)b * nchunks, nchunks, min(RB, W), S0,
                         cpow(args.lambda_bar[m], 64), (ep << 2) | FLAG_AGG, (ep << 2) | FLAG_INCL, hdr,
                         1000ull * (lim ? lim : 1000000u));
        }
    } else if (fits) {
        if (threadIdx.x == 0) {
            for (int s = 0; s < STAGES; ++s) {
                mbar_init(&sb->full_u[s], 1);
                mbar_init(&sb->empty_u[s], 2);     // the commits of GEMM1's two halves
            }
            for (int r = 0; r < REGIONS; ++r) {
                mbar_init(&sb->tmem_full[r], 2);   // the commits of GEMM1's two halves
                mbar_init(&sb->tmem_empty[r], 4);  // the four epilogue warps
                mbar_init(&sb->mma2_done[r], 2);   // the commits of GEMM2's two halves
            }
            mbar_init(&sb->xready, 4);             // the four scan warps
            mbar_init(&sb->xfree, 2);              // the commits of GEMM2's two halves
            mbar_init(&sb->eu_full, 1);
            mbar_init(&sb->eu_empty, 4);           // the four epilogue warps
            mbar_init(&sb->weights, 1);
            mbar_init(&sb->drain, 4);          // the four MMA-issuing threads
            for (int q = 0; q < 2; ++q) {
                mbar_init(&sb->carry_full[q], 4);    // the four fold warps
                mbar_init(&sb->carry_empty[q], 4);   // the four scan warps
            }
            sb->abort = 0;
            fence_mbar_init();
            griddep_wait();
            // epoch (word 3), drop_publish (4) and wait_limit_us (5) in two
            // independent 16-byte loads instead of three ordered ones
            const uint4 h0 = __ldcg(reinterpret_cast<const uint4 *>(hdr));
            const uint4 h1 = __ldcg(reinterpret_cast<const uint4 *>(hdr) + 1);
            sb->epoch = h0.w;
            sb->drop = h1.x;
            sb->limit_ns = 1000ull * (h1.y ? h1.y : 1000000u);
        }
        if (warp == W_TMEM) {
            tmem_alloc(&sb->tmem_base, 512);
            tmem_relinquish();
        }
    } else if (threadIdx.x == 0) {
        griddep_wait();
        latch_status(hdr, S5_ERR_UNSUPPORTED);
    }
    // barrier set-up and the TMEM allocation above overlap the end of the
    // kernel before this one; nothing global is touched before this wait
    griddep_wait();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const bool pipeline = fits && !scanner;
    const uint32_t tmem = pipeline ? sb->tmem_base : 0u;
    const unsigned tag = pipeline ? ((sb->epoch << 2) | FLAG_AGG) : 0u;

    if (!pipeline) {
        // nothing to run: straight to the teardown
    } else if (warp < 4) {
        // ------------------------------------------------------------ TMA and MMA issue
        // One thread in each of the four sub-partitions issues MMAs: warp 0
        // loads the u tiles and issues GEMM1's Re half, warp 1 GEMM1's Im
        // half, warps 2 and 3 the two K halves of GEMM2 (modes 0..63 and
        // 64..127).  A tensor pipe fed by one issuing thread slows down when
        // the FMA-bound warps of the same sub-partition compete for its issue
        // slots; spread over four, the issue keeps up with the pipe.
        if (lane == 0) {
            const uint32_t idesc = idesc_bf16_f32(128, T_TOK);
            const uint32_t bs = smem_addr(smem + SM_BS), cp = smem_addr(smem + SM_CP);
            const uint32_t xs = smem_addr(smem + SM_X);
            int issued = 0;   // u tiles 0 .. issued-1 have been requested
            // u tile il into stage il % STAGES once GEMM1 has read the tile before
            auto load_u = [&](int il) -> bool {
                const int s = il % STAGES;
                if (il >= STAGES && !pipe_wait(&sb->empty_u[s], ((il / STAGES) - 1) & 1, sb, hdr)) return false;
                int b, c;
                ln.tile(il, b, c);
#if S5_TC_REV
                c = nchunks - 1 - c;
#endif
                unsigned char *dst = smem + SM_U + s * U_STAGE;
                mbar_arrive_tx(&sb->full_u[s], U_STAGE);
                tma_load_3d(dst, &tmap_u, 0, c * T_TOK, b, &sb->full_u[s]);
                tma_load_3d(dst + T_TOK * 128, &tmap_u, 64, c * T_TOK, b, &sb->full_u[s]);
                issued = il + 1;
                return true;
            };
            bool ok = true;
            if (warp == 0) {
                prefetch_tmap(&tmap_u);
#if S5_TC_REV
                prefetch_tmap(&tmap_e);
#endif
                // the first u tiles come from HBM, the weight images from L2:
                // the longer latency is requested first
                for (int il = 0; il < n && il < STAGES; ++il) load_u(il);
                mbar_arrive_tx(&sb->weights, BS_BYTES + CP_BYTES);
                bulk_load(smem + SM_BS, args.ws.wimg + SM_BS, BS_BYTES, &sb->weights);
                bulk_load(smem + SM_CP, args.ws.wimg + SM_CP, CP_BYTES, &sb->weights);
            }
            ok = n == 0 || pipe_wait(&sb->weights, 0, sb, hdr);
            if (warp < 2) {
                // GEMM1 of tile g into region g % REGIONS: Re rows (warp 0)
                // into columns 0..63, Im rows (warp 1) into 64..127.
                const int mb = warp;
                const uint64_t da = sw128_kmajor_desc(bs);
                for (int g = 0; ok && g < n; ++g) {
                    const int s = g % STAGES, r = g % REGIONS;
                    ok = pipe_wait(&sb->full_u[s], (g / STAGES) & 1, sb, hdr) &&
                         (g < REGIONS || pipe_wait(&sb->tmem_empty[r], ((g / REGIONS) - 1) & 1, sb, hdr));
                    if (!ok) break;
                    tc_fence_after();
                    // descriptors: a base plus compile-time offsets (a descriptor's
                    // low bits hold the address / 16, and no offset carries out)
                    const uint64_t db = sw128_kmajor_desc(smem_addr(smem + SM_U + s * U_STAGE));
                    const uint64_t dam = da + (uint64_t)((mb * (P_M * 128)) >> 4);
                    const uint32_t d0 = tmem + (uint32_t)r * 128u + (uint32_t)mb * 64u;
#pragma unroll
                    for (int kq = 0; kq < H_F / 16; ++kq) {
                        const uint64_t a = dam + (uint64_t)(((kq >> 2) * (2 * P_M * 128) + (kq & 3) * 32) >> 4);
                        const uint64_t bb = db + (uint64_t)(((kq >> 2) * (T_TOK * 128) + (kq & 3) * 32) >> 4);
                        if (kq == 0)
                            mma_bf16_c<false>(d0, a, bb, idesc);
                        else
                            mma_bf16_c<true>(d0, a, bb, idesc);
                    }
                    mma_commit(&sb->tmem_full[r]);
                    mma_commit(&sb->empty_u[s]);
                    // warp 0 refills the stage tile g-1 used (its GEMM1 was
                    // issued an iteration ago) with tile g-1+STAGES
                    if (warp == 0 && g >= 1 && g - 1 + STAGES < n) ok = load_u(g - 1 + STAGES);
                }
            } else {
                // GEMM2 of tile g once X is complete (the scan warps have also
                // read the tile's Bu by then): warp 2 sums modes 0..63 into
                // columns 0..63 of the tile's region, warp 3 modes 64..127
                // into columns 64..127; the epilogue adds the two.
                const int kh = warp - 2;
                const uint64_t dc = sw128_kmajor_desc(cp), dx = sw128_kmajor_desc(xs);
                for (int g = 0; ok && g < n; ++g) {
                    const int r = g % REGIONS;
                    ok = pipe_wait(&sb->xready, g & 1, sb, hdr);
                    if (!ok) break;
                    tc_fence_after();
                    const uint32_t d = tmem + (uint32_t)r * 128u + (uint32_t)kh * 64u;
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk) {
                        const int kq = 8 * kh + kk;
                        const uint64_t a = dc + (uint64_t)(((kq >> 2) * (H_F * 128) + (kq & 3) * 32) >> 4);
                        const uint64_t bb = dx + (uint64_t)(((kq >> 2) * (T_TOK * 128) + (kq & 3) * 32) >> 4);
                        if (kk == 0)
                            mma_bf16_c<false>(d, a, bb, idesc);
                        else
                            mma_bf16_c<true>(d, a, bb, idesc);
                    }
                    mma_commit(&sb->xfree);
                    mma_commit(&sb->mma2_done[r]);
                }
            }
            // every MMA issued must complete before TMEM is freed
            mma_commit(&sb->drain);
            drain_wait(&sb->drain, 0);
            // copies still in flight must land before the CTA exits
            if (warp == 0) {
                drain_wait(&sb->weights, 0);
                for (int il = max(0, issued - STAGES); il < issued; ++il)
                    drain_wait(&sb->full_u[il % STAGES], (il / STAGES) & 1);
            }
        }
    } else if (warp >= W_SCAN && warp < W_SCAN + 4) {
        // ------------------------------------------------------------ scan
        const int qd = warp - W_SCAN;           // TMEM lane quarter = k-block of X
        const int m = 32 * qd + lane;
        ScanConsts kc;
        kc.lb = args.lambda_bar[m];
        kc.lb16 = cpow(kc.lb, 16);
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

        // Step j runs pass 1 of tile j, then pass 2 of tile j - 2.  The four
        // warps meet only through the pipeline's mbarriers (X complete, carry
        // slot read), each with its own count; a warp whose wait gave up leaves
        // the loop, and the abort flag it set ends the others' next waits.
        ScanTile t0, t1, t2;
        float2 xprev = make_float2(0.f, 0.f);
        bool mine = true;
        for (int j = 0; j < n + 2; ++j) {
            if (mine && j < n) mine = scan_front(t2, j, ln, L, lane_base, kc, rec, m, tag, drop, sb, hdr);
            if (!mine) break;
            const int i = j - 2;
            if (i >= 0) {
                // carry of tile i: from the carry warps' slot, or (one lane per
                // sequence) the previous tile's end state
                int b0, c0;
                ln.tile(i, b0, c0);
                const int r0 = i % REGIONS;
                float2 carry = xprev;
                if (W > 1) {
                    mine = pipe_wait(&sb->carry_full[i & 1], (i >> 1) & 1, sb, hdr);
                    if (mine) {
                        carry = slots[(i & 1) * P_M + m];
                        __syncwarp();
                        if (lane == 0) mbar_arrive(&sb->carry_empty[i & 1]);
                    }
                } else if (c0 == 0) {
                    carry = args.x0 ? args.x0[(size_t)b0 * P_M + m] : make_float2(0.f, 0.f);
                }
                // pass 2 once GEMM2 of tile i-1 has read X
                if (mine) mine = i == 0 || pipe_wait(&sb->xfree, (i - 1) & 1, sb, hdr);
                if (mine) {
                    tc_fence_after();
                    const uint32_t col0 = lane_base + (uint32_t)r0 * 128u;
                    xprev = (t0.Tc == T_TOK) ? pass2_full(col0, xb, kc, carry, t0.e)
                                             : pass2_short(col0, xb, kc.lb, carry, t0.Tc);
                    if (c0 == nchunks - 1 && args.x_last) args.x_last[(size_t)b0 * P_M + m] = xprev;
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
        // thread = feature h = TMEM lane of GEMM2: y = acc_lo + acc_hi + D * u
        // over the tile's tokens.  The tile's u is loaded before waiting for
        // GEMM2 and left untouched until after the wait (no instruction
        // depends on the loads before then), so their latency overlaps the
        // wait; the region is released once its last column is in registers.
        // Lane 0 of warp W_EPI keeps the u buffer filled: a second TMA load of
        // each tile's u, issued once all four warps have read the previous one.
        const int qd = warp - W_EPI;
        const int h = 32 * qd + lane;
#if S5_TC_REV
        const float dh = 1.f;   // the copy holds y, which is added
#else
        const float dh = args.d[h];
#endif
        const uint32_t lane_base = tmem + ((uint32_t)(32 * qd) << 16);
        unsigned short *yout = static_cast<unsigned short *>(args.y);
        // this feature's u for token t: row t, column h of the swizzled copy
        const unsigned char *eu = smem + SM_EU + (h >> 6) * (T_TOK * 128);
        const uint32_t hc = (uint32_t)(h & 63);
        const bool copier = qd == 0 && lane == 0;
        int eu_last = -1;
        auto load_eu = [&](int i) {
            int b, c;
            ln.tile(i, b, c);
            mbar_arrive_tx(&sb->eu_full, U_STAGE);
#if S5_TC_REV
            c = nchunks - 1 - c;
            tma_load_3d(smem + SM_EU, &tmap_e, 0, c * T_TOK, b, &sb->eu_full);
            tma_load_3d(smem + SM_EU + T_TOK * 128, &tmap_e, 64, c * T_TOK, b, &sb->eu_full);
#else
            tma_load_3d(smem + SM_EU, &tmap_u, 0, c * T_TOK, b, &sb->eu_full);
            tma_load_3d(smem + SM_EU + T_TOK * 128, &tmap_u, 64, c * T_TOK, b, &sb->eu_full);
#endif
            eu_last = i;
        };
        if (copier && n > 0) load_eu(0);
        for (int i = 0; i < n; ++i) {
            const int r = i % REGIONS;
            int b, c;
            ln.tile(i, b, c);
#if S5_TC_REV
            c = nchunks - 1 - c;
#endif
            const int Tc = min(T_TOK, L - c * T_TOK);
            const size_t row0 = ((size_t)b * L + (size_t)c * T_TOK) * H_F + h;
            unsigned short *yrow = yout + row0;
            // every exit is taken by the whole warp (the TMEM loads below are
            // warp-wide instructions)
            if (!__all_sync(0xffffffffu, pipe_wait(&sb->eu_full, i & 1, sb, hdr))) break;
            // tokens 2k and 2k+1 packed into uv[k] (low and high half)
            uint32_t uv[T_TOK / 2];
#pragma unroll
            for (int k = 0; k < T_TOK / 2; ++k) {
                const uint32_t lo = *reinterpret_cast<const unsigned short *>(
                    eu + (2 * k) * 128 + ((((hc >> 3) ^ (uint32_t)((2 * k) & 7))) << 4) + ((hc & 7u) << 1));
                const uint32_t hi = *reinterpret_cast<const unsigned short *>(
                    eu + (2 * k + 1) * 128 + ((((hc >> 3) ^ (uint32_t)((2 * k + 1) & 7))) << 4) + ((hc & 7u) << 1));
                uv[k] = lo | (hi << 16);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&sb->eu_empty);
            bool go = true;
            if (copier && i + 1 < n) {
                go = pipe_wait(&sb->eu_empty, i & 1, sb, hdr);
                if (go) load_eu(i + 1);
            }
            go = __shfl_sync(0xffffffffu, go, 0);
            if (!__all_sync(0xffffffffu, go && pipe_wait(&sb->mma2_done[r], (i / REGIONS) & 1, sb, hdr))) break;
            tc_fence_after();
#pragma unroll
            for (int hf = 0; hf < 4; ++hf) {
                uint32_t ya[16], yb[16];
                tmem_ld16(lane_base + (uint32_t)r * 128u + (uint32_t)hf * 16u, ya);
                tmem_ld16(lane_base + (uint32_t)r * 128u + 64u + (uint32_t)hf * 16u, yb);
                tmem_wait_ld();
                if (hf == 3) {
                    // every column of the region has been read: it may be reused
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&sb->tmem_empty[r]);
                }
#pragma unroll
                for (int k = 0; k < 16; ++k) {
                    const int t = hf * 16 + k;
                    const uint32_t ub = (t & 1) ? (uv[t >> 1] & 0xFFFF0000u) : (uv[t >> 1] << 16);
                    const float v = fmaf(dh, __uint_as_float(ub),
                                         __uint_as_float(ya[k]) + __uint_as_float(yb[k]));
                    if (t < Tc) yrow[(size_t)t * H_F] = __bfloat16_as_ushort(__float2bfloat16_rn(v));
                }
            }
        }
        // a copy still in flight (the loop left early) must land before the CTA exits
        if (copier && eu_last >= 0) drain_wait(&sb->eu_full, eu_last & 1);
    } else if (warp >= W_FOLD && warp < W_FOLD + 4 && W > 1) {
        // ------------------------------------------------------------ carries
        const int m = 32 * (warp - W_FOLD) + lane;
        float2 *slots = reinterpret_cast<float2 *>(smem + SM_CARRY);
        const float4 *carry = args.ws.carry;
        const unsigned tag_s = (sb->epoch << 2) | FLAG_INCL;
        const unsigned long long limit = sb->limit_ns;
        const int b = ln.kb, p = ln.kp;
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

// The bf16 images of B_bar and C' that the scan kernel bulk-copies in.
cudaError_t launch_weight_images(const TcArgs &a, cudaStream_t st) {
    const int words = P_M * H_F / 2 + H_F * P_M;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((words + 255) / 256));
    cfg.blockDim = dim3(256);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    set_programmatic(attr[0]);
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, weight_images_kernel, a.b_bar, a.c_tilde, a.ws.wimg);
}

}  // namespace

#if !S5_TC_REV
bool tc_supported(int H, int P, bool u_bf16, bool y_bf16, bool proj_bf16) {
    return H == H_F && P == P_M && u_bf16 && y_bf16 && proj_bf16;
}

// Lanes per sequence and grid: W lanes plus one scanner per sequence, B*(W+1)
// CTAs (2 <= W <= nchunks, W <= W_MAX), when at least three CTAs per sequence
// fit on the SMs; else W = 1, min(B, SMs) CTAs, each taking whole sequences.
// TC_FREE_SMS SMs stay out of the grid: the kernel launched after this one
// (programmatically) becomes resident there while this grid runs, so that
// its start -- instructions fetched into cold caches, its first loads --
// overlaps this kernel instead of following it.
void tc_grid(int B, int nchunks, int num_sms, int *W, int *G) {
    const int usable = num_sms > 2 * TC_FREE_SMS ? num_sms - TC_FREE_SMS : num_sms;
    int w = B <= usable ? usable / B - 1 : 0;
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
    cudaError_t e = launch_weight_images(a, st);
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
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    set_programmatic(attr[1]);
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, fwd_tc_kernel, mu, a);
}

#else
cudaError_t launch_backward_add_tc(const TcArgs &a0, const void *u, cudaStream_t st, int num_sms) {
    TcArgs a = a0;
    a.u = u;
    a.x0 = nullptr;
    a.x_last = nullptr;
    int G = 0;
    tc_grid(a.B, a.nchunks, num_sms, &a.W, &G);
    CUtensorMap mu, my;
    if (!make_map(&mu, u, a.B, a.L)) return cudaErrorInvalidValue;
    if (!make_map(&my, a.y, a.B, a.L)) return cudaErrorInvalidValue;
    cudaError_t e = launch_weight_images(a, st);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(bwd_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_REQUEST);
    if (e != cudaSuccess) return e;
    // cooperative launch, as for the forward scan
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, bwd_tc_kernel, THREADS, SMEM_REQUEST);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) return cudaErrorCooperativeLaunchTooLarge;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)G);
    cfg.blockDim = dim3(THREADS);
    cfg.dynamicSmemBytes = SMEM_REQUEST;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    set_programmatic(attr[1]);
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, bwd_tc_kernel, mu, my, a);
}
#endif

}  // namespace s5
