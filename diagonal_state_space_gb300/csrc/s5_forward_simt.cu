// s5_forward_simt.cu -- fused S5 forward on the CUDA cores (float32 FFMA).
//
// One CTA processes one tile: T consecutive tokens of one sequence and all P
// modes.  Per tile, entirely in shared memory and registers:
//   1. u tile -> smem (float32);
//   2. Bu[t][p] = sum_h W[p][h] u[t][h]   (W = B_bar, or B_tilde for irregular
//      sampling), register-tiled 4 tokens x 2 modes per thread;
//   3. the tile's own scan: each (mode, segment) thread folds its segment's
//      affine maps (a, b) from a zero start, then the segments are folded into
//      the tile aggregate (A, E) -- the associative operator of the review's
//      "Associative scans preserve the recurrence" / summary App. H:
//      (a1,b1) then (a2,b2) = (a2 a1, a2 b1 + b2);
//   4. decoupled look-back across tiles (Merrill & Garland, "Single-pass
//      Parallel Prefix Scan with Decoupled Look-back", 2016): publish (A, E),
//      fold predecessors' aggregates until an inclusive state is found,
//      publish this tile's inclusive state;
//   5. rerun the segments from their true carries, writing x_k in place;
//   6. y[t][h] = 2 sum_p Re(C[h][p] x[t][p]) + D[h] u[t][h], register-tiled
//      4 tokens x 4 features, then stored.
// Bu and x never leave the SM.  Tiles are claimed in order through an atomic
// counter, so every tile a CTA waits on is held by a running CTA.
#include "s5_simt.cuh"

namespace s5 {

constexpr int SIMT_THREADS = 256;
constexpr int SIMT_KC = 16;     // K-chunk of the staged weights
constexpr int SIMT_MAXMT = 4;   // register micro-tiles per thread

// 2*pi split for Cody-Waite reduction: 6.28125 is exact in 8 bits, so n*C0 is
// exact for the n that occur; C1 + C2 carry the rest of 2*pi to ~2^-61.
constexpr float TWO_PI_0 = 6.28125f;
constexpr float TWO_PI_1 = 0x1.fb5444p-10f;
constexpr float TWO_PI_2 = 0x1.68c234p-37f;
constexpr float INV_TWO_PI = 0.15915494f;

// Per-thread asynchronous copies (8 bytes) into shared memory: the staged
// weights of the next chunk load while the current chunk is computed.
__device__ __forceinline__ void cp_async8(void *smem_dst, const void *gsrc) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(
                     static_cast<uint32_t>(__cvta_generic_to_shared(smem_dst))),
                 "l"(gsrc)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

struct SimtSmem {
    int Pe, He, T;
    size_t u_off, x_off, a_off, w_off, seg_off, tagg_off, carry_off, g_off, total;
};

__host__ __device__ inline SimtSmem simt_smem(int T, int H, int P, int nseg, bool varying) {
    SimtSmem s;
    s.T = T;
    s.Pe = P + (P & 1);
    s.He = (H + 3) & ~3;
    size_t off = 0;
    auto take = [&](size_t bytes) { size_t o = off; off += (bytes + 15) & ~size_t(15); return o; };
    s.u_off = take(sizeof(float) * (size_t)T * H);
    s.x_off = take(sizeof(float2) * (size_t)T * s.Pe);
    s.a_off = take(varying ? sizeof(float2) * (size_t)T * s.Pe : 0);
    // two staged chunks of SIMT_KC weight rows, each row padded by two float2
    s.w_off = take(2 * sizeof(float2) * (size_t)SIMT_KC * ((s.Pe > s.He ? s.Pe : s.He) + 2));
    s.seg_off = take(sizeof(float4) * (size_t)nseg * P);
    s.tagg_off = take(sizeof(float4) * (size_t)P);
    s.carry_off = take(sizeof(float4) * (size_t)P);
    s.g_off = take(varying ? sizeof(float) * (size_t)T : 0);
    s.total = off;
    return s;
}

// Coefficients of one irregular step: a = exp(z), gain = (a-1)/lambda with
// z = g*lambda*Delta.  The phase g*Im(lambda)*Delta (up to a few hundred
// radians) is formed as an exact float pair and reduced modulo 2*pi before
// sincosf; Re(a-1) = expm1(x)cos(r) - (1 - cos r) keeps small steps accurate.
__device__ __forceinline__ void irregular_step(const ModeConst &m, float2 inv_lam, float g,
                                               float2 &a, float2 &gain) {
    float th = g * m.om_hi;
    float th_err = fmaf(g, m.om_hi, -th) + g * m.om_lo;
    float x = g * m.rho;
    if (g * m.zabs < 1e-4f) {
        // Delta_k * phi1(z), phi1(z) = 1 + z/2 + z^2/6 + z^3/24 (next term < 1e-18)
        float2 z = make_float2(x, th + th_err);
        float2 phi = make_float2(1.f / 24.f, 0.f);
        phi = cfma(phi, z, make_float2(1.f / 6.f, 0.f));
        phi = cfma(phi, z, make_float2(0.5f, 0.f));
        phi = cfma(phi, z, make_float2(1.f, 0.f));
        float dk = g * m.dt;
        gain = make_float2(dk * phi.x, dk * phi.y);
        // exp(z) = 1 + z*phi1(z)
        float2 zp = cmul(z, phi);
        a = make_float2(1.f + zp.x, zp.y);
        return;
    }
    float n = rintf(th * INV_TWO_PI);
    float r = fmaf(-n, TWO_PI_0, th);
    r = fmaf(-n, TWO_PI_1, r);
    r = fmaf(-n, TWO_PI_2, r);
    r += th_err;
    float sr, cr;
    sincosf(r, &sr, &cr);
    float em1 = expm1f(x);
    float mag = 1.f + em1;
    a = make_float2(mag * cr, mag * sr);
    float omc = cr > 0.f ? (sr * sr) / (1.f + cr) : 1.f - cr;   // 1 - cos r without cancellation
    float2 am1 = make_float2(fmaf(em1, cr, -omc), mag * sr);
    gain = cmul(am1, inv_lam);
}

// NT threads per CTA.
template <typename UT, typename YT, bool VARYING, int NT>
__global__ void __launch_bounds__(NT)
fwd_simt_kernel(const SimtArgs args) {
    extern __shared__ __align__(16) unsigned char smem[];
    __shared__ long long s_tile;
    __shared__ unsigned s_epoch, s_drop, s_bad;
    __shared__ unsigned s_st[32];   // look-back window: status of predecessors c-1, c-2, ...
    __shared__ int s_n, s_stop;
    __shared__ unsigned long long s_limit;

    const int tid = threadIdx.x;
    const int B = args.B, L = args.L, H = args.H, P = args.P, T = args.T, nseg = args.nseg;
    const SimtSmem lay = simt_smem(T, H, P, nseg, VARYING);
    const int Pe = lay.Pe, He = lay.He;
    float *u_s = reinterpret_cast<float *>(smem + lay.u_off);
    float2 *x_s = reinterpret_cast<float2 *>(smem + lay.x_off);
    float2 *a_s = reinterpret_cast<float2 *>(smem + lay.a_off);
    float2 *w_s = reinterpret_cast<float2 *>(smem + lay.w_off);
    // staged chunks: two buffers of SIMT_KC rows, refilled alternately
    // staged rows are padded by two float2: rows kk and kk+1 then start four
    // banks apart, so the transposing stores of a warp's 16 row indices meet
    // in pairs, not all in one bank, and rows stay 16-byte aligned
    const int PeS = Pe + 2, HeS = He + 2;
    const size_t wbuf_len = (size_t)SIMT_KC * ((Pe > He ? Pe : He) + 2);
    auto wbuf = [&](int k) { return w_s + (size_t)(k & 1) * wbuf_len; };
    // chunk [h0, h0 + SIMT_KC) of B_bar^T (rows kk, columns p) or C~^T
    auto stage_w = [&](float2 *dst, int h0) {
        const int kc = min(SIMT_KC, H - h0);
        for (int i = tid; i < Pe * SIMT_KC; i += NT) {
            const int p = i / SIMT_KC, kk = i - p * SIMT_KC;
            float2 *d = dst + kk * PeS + p;
            if (p < P && kk < kc)
                cp_async8(d, args.w + (size_t)p * H + h0 + kk);
            else
                *d = make_float2(0.f, 0.f);
        }
        cp_async_commit();
    };
    auto stage_c = [&](float2 *dst, int q0) {
        const int kc = min(SIMT_KC, P - q0);
        for (int i = tid; i < He * SIMT_KC; i += NT) {
            const int h = i / SIMT_KC, kk = i - h * SIMT_KC;
            float2 *d = dst + kk * HeS + h;
            if (h < H && kk < kc)
                cp_async8(d, args.c_tilde + (size_t)h * P + q0 + kk);
            else
                *d = make_float2(0.f, 0.f);
        }
        cp_async_commit();
    };
    float4 *seg_s = reinterpret_cast<float4 *>(smem + lay.seg_off);
    float4 *tagg_s = reinterpret_cast<float4 *>(smem + lay.tagg_off);
    float4 *carry_s = reinterpret_cast<float4 *>(smem + lay.carry_off);
    float *g_s = reinterpret_cast<float *>(smem + lay.g_off);

    WsHeader *hdr = args.ws.hdr;
    if (tid == 0) {
        s_epoch = *reinterpret_cast<volatile unsigned *>(&hdr->epoch);
        s_drop = *reinterpret_cast<volatile unsigned *>(&hdr->drop_publish);
        unsigned lim = *reinterpret_cast<volatile unsigned *>(&hdr->wait_limit_us);
        s_limit = 1000ull * (lim ? lim : 1000000u);
        s_bad = 0;
    }
    const UT *u = static_cast<const UT *>(args.u);
    YT *y = static_cast<YT *>(args.y);
    const int PQ = (P + 1) / 2, HQ = (H + 3) / 4;
    const int nmt1 = (T / 4) * PQ, nmt2 = (T / 4) * HQ;

    for (;;) {
        __syncthreads();
        if (tid == 0) s_tile = (long long)atomicAdd(&hdr->tile_counter, 1u);
        __syncthreads();
        const long long tile = s_tile;
        if (tile >= args.ntiles) break;
        const unsigned epoch = s_epoch;
        const bool publish = s_drop != (unsigned)(tile + 1);
        const int b = (int)(tile % B);
        const int c = (int)(tile / B);
        const int t0 = c * T;
        const int Tc = min(T, L - t0);

        // the first weight chunk loads while the u tile does (the barriers at
        // the loop top follow every read of the buffers by the tile before)
        stage_w(wbuf(0), 0);

        // 1. input tile (zero rows past the ragged end)
        const size_t row0 = (size_t)b * L + t0;
        for (int i = tid; i < T * H; i += NT) {
            int t = i / H, h = i - t * H;
            u_s[i] = t < Tc ? load_elem<UT>(u + (row0 + t) * H + h) : 0.f;
        }
        if (VARYING) {
            for (int t = tid; t < T; t += NT) {
                float gv = 0.f;
                if (t < Tc) {
                    gv = __ldg(args.g + row0 + t);
                    if (!(gv >= 0.f) || !isfinite(gv)) { s_bad = 1; gv = 0.f; }
                }
                g_s[t] = gv;
            }
        }

        // 2. input projection Bu = W u (K-loop over features in chunks of SIMT_KC)
        {
            float acc[SIMT_MAXMT][4][4];
#pragma unroll
            for (int m = 0; m < SIMT_MAXMT; ++m)
#pragma unroll
                for (int i = 0; i < 4; ++i)
#pragma unroll
                    for (int j = 0; j < 4; ++j) acc[m][i][j] = 0.f;
            for (int h0 = 0, ci = 0; h0 < H; h0 += SIMT_KC, ++ci) {
                const int kc = min(SIMT_KC, H - h0);
                // chunk ci+1 into the other buffer (read two chunks ago,
                // released by the barrier ending that chunk), then chunk ci
                if (h0 + SIMT_KC < H) {
                    stage_w(wbuf(ci + 1), h0 + SIMT_KC);
                    cp_async_wait<1>();
                } else {
                    cp_async_wait<0>();
                }
                __syncthreads();   // chunk ci (and, the first time, the u tile) is complete
                const float2 *wk = wbuf(ci);
#pragma unroll
                for (int m = 0; m < SIMT_MAXMT; ++m) {
                    const int mt = tid + m * NT;
                    if (mt < nmt1) {
                        const int pq = mt % PQ, tq = mt / PQ;
                        const float *ur = u_s + (size_t)(4 * tq) * H + h0;
                        const float4 *wr = reinterpret_cast<const float4 *>(wk + 2 * pq);
                        for (int kk = 0; kk < kc; ++kk) {
                            float4 wv = wr[kk * (PeS / 2)];
#pragma unroll
                            for (int i = 0; i < 4; ++i) {
                                float uv = ur[i * H + kk];
                                acc[m][i][0] = fmaf(wv.x, uv, acc[m][i][0]);
                                acc[m][i][1] = fmaf(wv.y, uv, acc[m][i][1]);
                                acc[m][i][2] = fmaf(wv.z, uv, acc[m][i][2]);
                                acc[m][i][3] = fmaf(wv.w, uv, acc[m][i][3]);
                            }
                        }
                    }
                }
                __syncthreads();   // every thread is done with this chunk's buffer
            }
#pragma unroll
            for (int m = 0; m < SIMT_MAXMT; ++m) {
                const int mt = tid + m * NT;
                if (mt < nmt1) {
                    const int pq = mt % PQ, tq = mt / PQ;
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        *reinterpret_cast<float4 *>(x_s + (size_t)(4 * tq + i) * Pe + 2 * pq) =
                            make_float4(acc[m][i][0], acc[m][i][1], acc[m][i][2], acc[m][i][3]);
                }
            }
        }
        __syncthreads();
        // the readout's first weight chunk loads during the scan
        stage_c(wbuf(0), 0);

        // 3. per-segment fold, from a zero start
        const int seglen = (Tc + nseg - 1) / nseg;
        for (int i = tid; i < P * nseg; i += NT) {
            const int p = i % P, s = i / P;
            const int s0 = min(Tc, s * seglen), s1 = min(Tc, s0 + seglen);
            float2 A = make_float2(1.f, 0.f), E = make_float2(0.f, 0.f);
            if (!VARYING) {
                const float2 lb = args.lambda_bar[p];
                for (int t = s0; t < s1; ++t) {
                    E = cfma(lb, E, x_s[(size_t)t * Pe + p]);
                    A = cmul(lb, A);
                }
            } else {
                const ModeConst mc = args.ws.modes[p];
                const float2 inv = make_float2(mc.inv_re, mc.inv_im);
                for (int t = s0; t < s1; ++t) {
                    float2 a, gain;
                    irregular_step(mc, inv, g_s[t], a, gain);
                    const size_t k = (size_t)t * Pe + p;
                    const float2 bk = cmul(gain, x_s[k]);
                    x_s[k] = bk;
                    a_s[k] = a;
                    E = cfma(a, E, bk);
                    A = cmul(a, A);
                }
            }
            seg_s[(size_t)s * P + p] = make_float4(A.x, A.y, E.x, E.y);
        }
        __syncthreads();

        // 4. tile aggregate, publication and look-back
        for (int p = tid; p < P; p += NT) {
            float2 A = make_float2(1.f, 0.f), E = make_float2(0.f, 0.f);
            for (int s = 0; s < nseg; ++s) {
                const float4 v = seg_s[(size_t)s * P + p];
                const float2 As = make_float2(v.x, v.y);
                E = cfma(As, E, make_float2(v.z, v.w));
                A = cmul(As, A);
            }
            tagg_s[p] = make_float4(A.x, A.y, E.x, E.y);
            if (c > 0) __stcg(args.ws.agg + tile * P + p, make_float4(A.x, A.y, E.x, E.y));
            float2 x0v = make_float2(0.f, 0.f);
            if (c == 0 && args.x0) x0v = args.x0[(size_t)b * P + p];
            carry_s[p] = make_float4(1.f, 0.f, x0v.x, x0v.y);
        }
        __syncthreads();
        if (c > 0) {
            if (tid == 0 && publish) {
                __threadfence();
                st_release(args.ws.flags + tile, (epoch << 2) | FLAG_AGG);
            }
            // Warp-wide look-back: lane l of warp 0 waits for predecessor
            // chunk jn - l (nearest first) to publish at least its aggregate;
            // a ballot finds the nearest one that is inclusive (or gave up).
            // The block then folds that whole window at once, nearest first,
            // and moves 32 chunks back only if every one was an aggregate.
            for (int jn = c - 1;; jn -= 32) {
                if (tid < 32) {
                    const int j = jn - tid;
                    unsigned st = 0;
                    if (j >= 0) st = wait_flag(hdr, args.ws.flags + (long long)j * B + b, epoch, s_limit, (unsigned)tile);
                    const unsigned stop = __ballot_sync(0xffffffffu, j < 0 || st != FLAG_AGG);
                    s_st[tid] = st;
                    if (tid == 0) {
                        s_n = stop ? __ffs(stop) : 32;
                        s_stop = stop != 0;
                    }
                }
                __syncthreads();
                const int n = s_n;
                for (int p = tid; p < P; p += NT) {
                    float4 cs = carry_s[p];
                    float2 mult = make_float2(cs.x, cs.y), accv = make_float2(cs.z, cs.w);
                    for (int l0 = 0; l0 < n; l0 += 8) {
                        float4 v[8];
#pragma unroll
                        for (int q = 0; q < 8; ++q) {
                            const int l = l0 + q;
                            v[q] = make_float4(1.f, 0.f, 0.f, 0.f);
                            if (l < n) {
                                const long long jt = (long long)(jn - l) * B + b;
                                if (s_st[l] == FLAG_AGG) {
                                    v[q] = __ldcg(args.ws.agg + jt * P + p);
                                } else if (s_st[l] == FLAG_INCL) {
                                    const float2 inc = __ldcg(args.ws.incl + jt * P + p);
                                    v[q] = make_float4(0.f, 0.f, inc.x, inc.y);
                                }
                            }
                        }
#pragma unroll
                        for (int q = 0; q < 8; ++q) {
                            const int l = l0 + q;
                            if (l < n && (s_st[l] == FLAG_AGG || s_st[l] == FLAG_INCL)) {
                                // aggregate (A, E): acc += mult E, mult *= A; inclusive: acc += mult x
                                accv = cfma(mult, make_float2(v[q].z, v[q].w), accv);
                                mult = cmul(mult, make_float2(v[q].x, v[q].y));
                            }
                        }
                    }
                    carry_s[p] = make_float4(mult.x, mult.y, accv.x, accv.y);
                }
                __syncthreads();
                if (s_stop) break;
            }
        }
        for (int p = tid; p < P; p += NT) {
            const float4 ta = tagg_s[p];
            const float4 cs = carry_s[p];
            const float2 inc = cfma(make_float2(ta.x, ta.y), make_float2(cs.z, cs.w),
                                    make_float2(ta.z, ta.w));
            __stcg(args.ws.incl + tile * P + p, inc);
            if (c == args.nchunks - 1 && args.x_last) args.x_last[(size_t)b * P + p] = inc;
        }
        __syncthreads();
        if (tid == 0 && publish) {
            __threadfence();
            st_release(args.ws.flags + tile, (epoch << 2) | FLAG_INCL);
        }

        // 5. rerun every segment from its true carry, x_k in place of b_k
        for (int i = tid; i < P * nseg; i += NT) {
            const int p = i % P, s = i / P;
            const int s0 = min(Tc, s * seglen), s1 = min(Tc, s0 + seglen);
            const float4 cs = carry_s[p];
            float2 x = make_float2(cs.z, cs.w);
            for (int q = 0; q < s; ++q) {
                const float4 v = seg_s[(size_t)q * P + p];
                x = cfma(make_float2(v.x, v.y), x, make_float2(v.z, v.w));
            }
            if (!VARYING) {
                const float2 lb = args.lambda_bar[p];
                for (int t = s0; t < s1; ++t) {
                    const size_t k = (size_t)t * Pe + p;
                    x = cfma(lb, x, x_s[k]);
                    x_s[k] = x;
                }
            } else {
                for (int t = s0; t < s1; ++t) {
                    const size_t k = (size_t)t * Pe + p;
                    x = cfma(a_s[k], x, x_s[k]);
                    x_s[k] = x;
                }
            }
        }

        // 6. readout y = 2 Re(C x) + D u
        {
            float acc[SIMT_MAXMT][4][4];
#pragma unroll
            for (int m = 0; m < SIMT_MAXMT; ++m)
#pragma unroll
                for (int i = 0; i < 4; ++i)
#pragma unroll
                    for (int j = 0; j < 4; ++j) acc[m][i][j] = 0.f;
            for (int q0 = 0, ci = 0; q0 < P; q0 += SIMT_KC, ++ci) {
                const int kc = min(SIMT_KC, P - q0);
                if (q0 + SIMT_KC < P) {
                    stage_c(wbuf(ci + 1), q0 + SIMT_KC);
                    cp_async_wait<1>();
                } else {
                    cp_async_wait<0>();
                }
                __syncthreads();   // chunk ci (and, the first time, x) is complete
                const float2 *ck = wbuf(ci);
#pragma unroll
                for (int m = 0; m < SIMT_MAXMT; ++m) {
                    const int mt = tid + m * NT;
                    if (mt < nmt2) {
                        const int hq = mt % HQ, tq = mt / HQ;
                        const float2 *xr = x_s + (size_t)(4 * tq) * Pe + q0;
                        const float4 *cr = reinterpret_cast<const float4 *>(ck + 4 * hq);
                        for (int kk = 0; kk < kc; ++kk) {
                            const float4 c01 = cr[kk * (HeS / 2)];
                            const float4 c23 = cr[kk * (HeS / 2) + 1];
#pragma unroll
                            for (int i = 0; i < 4; ++i) {
                                const float2 xv = xr[(size_t)i * Pe + kk];
                                acc[m][i][0] = fmaf(c01.x, xv.x, fmaf(-c01.y, xv.y, acc[m][i][0]));
                                acc[m][i][1] = fmaf(c01.z, xv.x, fmaf(-c01.w, xv.y, acc[m][i][1]));
                                acc[m][i][2] = fmaf(c23.x, xv.x, fmaf(-c23.y, xv.y, acc[m][i][2]));
                                acc[m][i][3] = fmaf(c23.z, xv.x, fmaf(-c23.w, xv.y, acc[m][i][3]));
                            }
                        }
                    }
                }
                __syncthreads();   // every thread is done with this chunk's buffer
            }
#pragma unroll
            for (int m = 0; m < SIMT_MAXMT; ++m) {
                const int mt = tid + m * NT;
                if (mt < nmt2) {
                    const int hq = mt % HQ, tq = mt / HQ;
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const int t = 4 * tq + i;
                        if (t >= Tc) continue;
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            const int h = 4 * hq + j;
                            if (h < H) {
                                const float v = fmaf(2.f, acc[m][i][j], __ldg(args.d + h) * u_s[(size_t)t * H + h]);
                                store_elem<YT>(y + (row0 + t) * H + h, v);
                            }
                        }
                    }
                }
            }
        }
    }

    // launch epilogue: the last CTA resets the counters and advances the epoch
    __syncthreads();
    if (tid == 0) {
        if (VARYING && s_bad) latch_status(hdr, S5_ERR_NONFINITE);
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

// ---------------------------------------------------------------------------
// Host side.
// ---------------------------------------------------------------------------
int simt_nseg(int P) {
    if (P > SIMT_THREADS) return 1;
    int n = SIMT_THREADS / P;
    return n > 8 ? 8 : n;
}

// Largest tile (tokens) that fits the register tiling and shared memory.
int simt_tile_tokens(int H, int P, bool varying) {
    const int PQ = (P + 1) / 2, HQ = (H + 3) / 4;
    for (int T = 64; T >= 4; T /= 2) {
        if ((T / 4) * PQ > SIMT_MAXMT * SIMT_THREADS) continue;
        if ((T / 4) * HQ > SIMT_MAXMT * SIMT_THREADS) continue;
        if (simt_smem(T, H, P, simt_nseg(P), varying).total > 220 * 1024) continue;
        return T;
    }
    return 0;
}

constexpr int SIMT_BIG_THREADS = 512;

template <typename UT, typename YT, bool V, int NT>
static cudaError_t launch_k(const SimtArgs &a, cudaStream_t st, int num_sms) {
    const size_t smem = simt_smem(a.T, a.H, a.P, a.nseg, V).total;
    auto kern = fwd_simt_kernel<UT, YT, V, NT>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, NT, smem);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) return cudaErrorInvalidConfiguration;
    long long grid = (long long)per_sm * num_sms;
    if (grid > a.ntiles) grid = a.ntiles;
    kern<<<(unsigned)grid, NT, smem, st>>>(a);
    return cudaGetLastError();
}

// Twice the warps when a single CTA fills an SM's shared memory.
template <typename UT, typename YT, bool V>
static cudaError_t launch_t(const SimtArgs &a, cudaStream_t st, int num_sms) {
    if (simt_smem(a.T, a.H, a.P, a.nseg, V).total > 112 * 1024)
        return launch_k<UT, YT, V, SIMT_BIG_THREADS>(a, st, num_sms);
    return launch_k<UT, YT, V, SIMT_THREADS>(a, st, num_sms);
}

cudaError_t launch_forward_simt(const SimtArgs &a, bool u_bf16, bool y_bf16, bool varying,
                                cudaStream_t st, int num_sms) {
    using bf = __nv_bfloat16;
    if (varying) {
        if (!u_bf16 && !y_bf16) return launch_t<float, float, true>(a, st, num_sms);
        if (!u_bf16 && y_bf16) return launch_t<float, bf, true>(a, st, num_sms);
        if (u_bf16 && !y_bf16) return launch_t<bf, float, true>(a, st, num_sms);
        return launch_t<bf, bf, true>(a, st, num_sms);
    }
    if (!u_bf16 && !y_bf16) return launch_t<float, float, false>(a, st, num_sms);
    if (!u_bf16 && y_bf16) return launch_t<float, bf, false>(a, st, num_sms);
    if (u_bf16 && !y_bf16) return launch_t<bf, float, false>(a, st, num_sms);
    return launch_t<bf, bf, false>(a, st, num_sms);
}

}  // namespace s5
