// s5_step.cu -- the streaming step and the helpers of the bidirectional layer.
//
// Streaming step (review "S5: Simplified State Space Layers for Sequence
// Modeling", "Associative scans preserve the recurrence": streaming inference
// keeps just the current state per layer; summary "SIMPLIFIED STATE SPACE
// LAYERS ...", App. C.1, online generation):
//   x <- lambda_bar * x + B_bar u,   y = 2 Re(C~ x) + D u.
// One cluster of 16 CTAs per group of up to 8 sequences.  CTA r owns a
// sixteenth of the modes: it reads its rows of B_bar once for all the group's
// sequences and updates their states; after a cluster barrier every CTA
// gathers the new states of all modes from its peers' shared memory
// (distributed shared memory) and forms the readout for its sixteenth of the
// features.  So B_bar and C~ are each read once per group rather than once per
// sequence, and every global load a warp needs is issued before any is used.
//
// Bidirectional layer ("Simplified State Space Layers for Sequence Modeling",
// "Paper vs code": a forward and a backward scan, C~ with 2P columns): the
// helpers split C~ into its two [H,P] halves, reverse sequences in time and add
// a time-reversed result into y.
#include <cooperative_groups.h>
#include <cuda_bf16.h>

#include "s5_internal.cuh"

namespace s5 {
namespace {

constexpr int STEP_THREADS = 512;
constexpr int STEP_CL = 16;   // CTAs per cluster (a non-portable size)
constexpr int STEP_SEQ = 8;   // sequences per cluster
constexpr int STEP_KC = 4;    // row elements per lane fetched up front (rows of up to 128)

// Sums each of N (a power of two, 2..32) per-lane values over the warp.  Each
// exchange halves the values a lane holds: the lane keeps the half its lane
// bit selects and adds its partner's copy of that half.  Afterwards lane l
// holds the total of value l / (32 / N) (the 32 / N lanes of a group agree).
template <int N>
__device__ __forceinline__ float warp_sum_many(float (&v)[N]) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int half = N / 2, o = 16; half >= 1; half /= 2, o /= 2) {
        const bool up = (lane & o) != 0;
#pragma unroll
        for (int j = 0; j < half; ++j) {
            const float keep = up ? v[j + half] : v[j];
            const float send = up ? v[j] : v[j + half];
            v[j] = keep + __shfl_xor_sync(0xffffffffu, send, o);
        }
    }
    float t = v[0];
#pragma unroll
    for (int o = 16 / N; o >= 1; o /= 2) t += __shfl_xor_sync(0xffffffffu, t, o);
    return t;
}

// Warp w of a CTA takes modes p0 + w, p0 + w + 16, ... and features h0 + w,
// h0 + w + 16, ...; for its first mode and feature every lane fetches its
// elements of the B_bar and C~ rows (and the states, lambda_bar, D) before
// anything else, so that one memory round trip covers them all.
__global__ void __launch_bounds__(STEP_THREADS, 1)
step_cluster_kernel(const float2 *__restrict__ lambda_bar, const float2 *__restrict__ b_bar,
                    const float2 *__restrict__ c_tilde, const float *__restrict__ d, float2 *__restrict__ x,
                    const float *__restrict__ u, float *__restrict__ y, int B, int H, int P) {
    namespace cg = cooperative_groups;
    cg::cluster_group cl = cg::this_cluster();
    const int r = (int)cl.block_rank();
    const int s0 = (int)(blockIdx.x / STEP_CL) * STEP_SEQ;
    const int ns = min(STEP_SEQ, B - s0);
    const int mp = (P + STEP_CL - 1) / STEP_CL, hp = (H + STEP_CL - 1) / STEP_CL;
    const int p0 = r * mp, p1 = min(P, p0 + mp), h0 = r * hp, h1 = min(H, h0 + hp);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
    extern __shared__ float2 sm_step[];
    float2 *sx_own = sm_step;                                // [STEP_SEQ][mp]: this CTA's new states
    float2 *sx_all = sx_own + STEP_SEQ * mp;                 // [STEP_SEQ][P]: every mode's new state
    float *su = reinterpret_cast<float *>(sx_all + STEP_SEQ * P);   // [STEP_SEQ][H]

    // nothing is read before the previous kernel in the stream (the step
    // before, which writes x) ends; then the next step may be scheduled
    griddep_wait();
    griddep_launch_dependents();

    // everything the first mode and feature of this warp need, fetched at once
    const int pf = p0 + warp, hf = h0 + warp;
    float2 bw[STEP_KC], cw[STEP_KC];
#pragma unroll
    for (int k = 0; k < STEP_KC; ++k) {
        const int h = lane + 32 * k, p = lane + 32 * k;
        bw[k] = (pf < p1 && h < H) ? b_bar[(size_t)pf * H + h] : make_float2(0.f, 0.f);
        cw[k] = (hf < h1 && p < P) ? c_tilde[(size_t)hf * P + p] : make_float2(0.f, 0.f);
    }
    float2 xo = make_float2(0.f, 0.f), lb = make_float2(0.f, 0.f);
    if (pf < p1 && lane < ns) {
        xo = x[(size_t)(s0 + lane) * P + pf];
        lb = lambda_bar[pf];
    }
    const float dh = hf < h1 ? d[hf] : 0.f;
    for (int i = threadIdx.x; i < ns * H; i += blockDim.x) su[i] = u[(size_t)s0 * H + i];
    __syncthreads();

    // input projection, a warp per mode, all sequences at once
    for (int p = pf; p < p1; p += nwarps) {
        const bool first = p == pf;
        float re[STEP_SEQ], im[STEP_SEQ];
#pragma unroll
        for (int q = 0; q < STEP_SEQ; ++q) re[q] = im[q] = 0.f;
        for (int h = lane, k = 0; h < H; h += 32, ++k) {
            float2 w;
            if (first && k < STEP_KC) {
                w = bw[0];
#pragma unroll
                for (int kk = 1; kk < STEP_KC; ++kk)
                    if (k == kk) w = bw[kk];
            } else {
                w = b_bar[(size_t)p * H + h];
            }
#pragma unroll
            for (int q = 0; q < STEP_SEQ; ++q)
                if (q < ns) {
                    const float v = su[q * H + h];
                    re[q] = fmaf(w.x, v, re[q]);
                    im[q] = fmaf(w.y, v, im[q]);
                }
        }
        // values 0..7: Re for the eight sequences, 8..15: Im; lane 2j holds value j
        float v[2 * STEP_SEQ];
#pragma unroll
        for (int q = 0; q < STEP_SEQ; ++q) {
            v[q] = re[q];
            v[STEP_SEQ + q] = im[q];
        }
        const float tot = warp_sum_many(v);
        const float bre = __shfl_sync(0xffffffffu, tot, 2 * lane);
        const float bim = __shfl_sync(0xffffffffu, tot, 2 * (STEP_SEQ + lane) & 31);
        if (lane < ns) {
            float2 xv = xo, lv = lb;
            if (!first) {
                xv = x[(size_t)(s0 + lane) * P + p];
                lv = lambda_bar[p];
            }
            sx_own[lane * mp + (p - p0)] =
                make_float2(fmaf(lv.x, xv.x, fmaf(-lv.y, xv.y, bre)), fmaf(lv.x, xv.y, fmaf(lv.y, xv.x, bim)));
        }
    }
    // the barrier releases only shared-memory writes: the states go to global
    // memory after it, so that it does not wait for those stores
    cl.sync();
    for (int i = threadIdx.x; i < ns * (p1 - p0); i += blockDim.x) {
        const int q = i / (p1 - p0), pl = i - q * (p1 - p0);
        x[(size_t)(s0 + q) * P + p0 + pl] = sx_own[q * mp + pl];
    }
    // every mode's new state, from the CTA that owns it
    for (int i = threadIdx.x; i < ns * P; i += blockDim.x) {
        const int q = i / P, p = i - q * P, owner = p / mp;
        const float2 *peer = cl.map_shared_rank(sx_own, owner);
        sx_all[q * P + p] = peer[q * mp + (p - owner * mp)];
    }
    __syncthreads();
    // readout, a warp per feature
    for (int h = hf; h < h1; h += nwarps) {
        const bool first = h == hf;
        float acc[STEP_SEQ];
#pragma unroll
        for (int q = 0; q < STEP_SEQ; ++q) acc[q] = 0.f;
        for (int p = lane, k = 0; p < P; p += 32, ++k) {
            float2 c;
            if (first && k < STEP_KC) {
                c = cw[0];
#pragma unroll
                for (int kk = 1; kk < STEP_KC; ++kk)
                    if (k == kk) c = cw[kk];
            } else {
                c = c_tilde[(size_t)h * P + p];
            }
#pragma unroll
            for (int q = 0; q < STEP_SEQ; ++q)
                if (q < ns) {
                    const float2 xv = sx_all[q * P + p];
                    acc[q] = fmaf(c.x, xv.x, fmaf(-c.y, xv.y, acc[q]));
                }
        }
        // lane 4q holds sequence q's sum
        const float mine = __shfl_sync(0xffffffffu, warp_sum_many(acc), (4 * lane) & 31);
        if (lane < ns) y[(size_t)(s0 + lane) * H + h] = fmaf(first ? dh : d[h], su[lane * H + h], 2.f * mine);
    }
    // no CTA leaves while a peer may still read its states (their reads are
    // complete once used, so the arrival need not order any memory access)
    asm volatile("barrier.cluster.arrive.relaxed.aligned;\n\tbarrier.cluster.wait.aligned;" ::: "memory");
}

// c2 [H][2P] -> cf [H][P] (columns 0..P-1), cb [H][P] (columns P..2P-1)
__global__ void split_c_kernel(const float2 *__restrict__ c2, int H, int P, float2 *__restrict__ cf,
                               float2 *__restrict__ cb) {
    const long long n = (long long)H * P;
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x) {
        const long long h = i / P, p = i % P;
        cf[i] = c2[h * 2 * P + p];
        cb[i] = c2[h * 2 * P + P + p];
    }
}

// dst[b][L-1-k][:] = src[b][k][:], rows of `row` elements of type T (T is a
// 16-byte vector where the row allows it); 32-bit indices, the launcher checks
// that B*L*row fits.
template <typename T>
__global__ void reverse_time_kernel(const T *__restrict__ src, T *__restrict__ dst, int B, int L, int row) {
    const unsigned n = (unsigned)B * L * row;
    for (unsigned i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) {
        const unsigned bk = i / row, e = i - bk * row, b = bk / L, k = bk - b * L;
        dst[((size_t)b * L + (L - 1 - k)) * row + e] = src[i];
    }
}

__device__ __forceinline__ float4 add4(float4 a, float4 b) {
    return make_float4(a.x + b.x, a.y + b.y, a.z + b.z, a.w + b.w);
}
__device__ __forceinline__ float2 f2_of(unsigned w) {
    return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&w));
}
__device__ __forceinline__ unsigned w_of(float2 f) {
    const __nv_bfloat162 h = __float22bfloat162_rn(f);
    return *reinterpret_cast<const unsigned *>(&h);
}
__device__ __forceinline__ uint4 add4(uint4 a, uint4 b) {  // 8 bf16, added in fp32, rounded once
    const float2 a0 = f2_of(a.x), a1 = f2_of(a.y), a2 = f2_of(a.z), a3 = f2_of(a.w);
    const float2 b0 = f2_of(b.x), b1 = f2_of(b.y), b2 = f2_of(b.z), b3 = f2_of(b.w);
    return make_uint4(w_of(make_float2(a0.x + b0.x, a0.y + b0.y)), w_of(make_float2(a1.x + b1.x, a1.y + b1.y)),
                      w_of(make_float2(a2.x + b2.x, a2.y + b2.y)), w_of(make_float2(a3.x + b3.x, a3.y + b3.y)));
}
__device__ __forceinline__ float add4(float a, float b) { return a + b; }
__device__ __forceinline__ __nv_bfloat16 add4(__nv_bfloat16 a, __nv_bfloat16 b) {
    return __float2bfloat16_rn(__bfloat162float(a) + __bfloat162float(b));
}

// y[b][k][:] += yr[b][L-1-k][:], rows of `row` elements of type T
template <typename T>
__global__ void add_reversed_kernel(T *__restrict__ y, const T *__restrict__ yr, int B, int L, int row) {
    const unsigned n = (unsigned)B * L * row;
    for (unsigned i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) {
        const unsigned bk = i / row, e = i - bk * row, b = bk / L, k = bk - b * L;
        y[i] = add4(y[i], yr[((size_t)b * L + (L - 1 - k)) * row + e]);
    }
}

int grid_for(long long n) {
    long long g = (n + 255) / 256;
    if (g > 152 * 16) g = 152 * 16;
    return g < 1 ? 1 : (int)g;
}

}  // namespace

size_t step_smem_bytes(int H, int P) {
    const size_t mp = (size_t)(P + STEP_CL - 1) / STEP_CL;
    return sizeof(float2) * STEP_SEQ * (mp + (size_t)P) + sizeof(float) * STEP_SEQ * (size_t)H;
}

cudaError_t launch_step(const float2 *lambda_bar, const float2 *b_bar, const float2 *c_tilde, const float *d,
                        float2 *x, const float *u, float *y, int B, int H, int P, cudaStream_t st) {
    const size_t smem = step_smem_bytes(H, P);
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(step_cluster_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
    }
    cudaError_t e = cudaFuncSetAttribute(step_cluster_kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
    const int clusters = (B + STEP_SEQ - 1) / STEP_SEQ;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(clusters * STEP_CL));
    cfg.blockDim = dim3(STEP_THREADS);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = STEP_CL;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    set_programmatic(attr[1]);
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, step_cluster_kernel, lambda_bar, b_bar, c_tilde, d, x, u, y, B, H, P);
}

cudaError_t launch_split_c(const float2 *c2, int H, int P, float2 *cf, float2 *cb, cudaStream_t st) {
    split_c_kernel<<<grid_for((long long)H * P), 256, 0, st>>>(c2, H, P, cf, cb);
    return cudaGetLastError();
}

cudaError_t launch_reverse_time(const void *src, void *dst, int B, int L, int H, int elem_bytes, cudaStream_t st) {
    const size_t row_bytes = (size_t)H * elem_bytes;
    if ((size_t)B * L * H >= (1ull << 31)) return cudaErrorInvalidValue;
    if (row_bytes % 16 == 0) {
        const int row = (int)(row_bytes / 16);
        reverse_time_kernel<uint4><<<grid_for((long long)B * L * row), 256, 0, st>>>(
            static_cast<const uint4 *>(src), static_cast<uint4 *>(dst), B, L, row);
    } else if (elem_bytes == 2) {
        reverse_time_kernel<unsigned short><<<grid_for((long long)B * L * H), 256, 0, st>>>(
            static_cast<const unsigned short *>(src), static_cast<unsigned short *>(dst), B, L, H);
    } else {
        reverse_time_kernel<float><<<grid_for((long long)B * L * H), 256, 0, st>>>(
            static_cast<const float *>(src), static_cast<float *>(dst), B, L, H);
    }
    return cudaGetLastError();
}

cudaError_t launch_add_reversed(void *y, const void *yr, int B, int L, int H, bool bf16, cudaStream_t st) {
    if ((size_t)B * L * H >= (1ull << 31)) return cudaErrorInvalidValue;
    const long long rows = (long long)B * L;
    if (bf16 && H % 8 == 0)
        add_reversed_kernel<uint4><<<grid_for(rows * (H / 8)), 256, 0, st>>>(
            static_cast<uint4 *>(y), static_cast<const uint4 *>(yr), B, L, H / 8);
    else if (bf16)
        add_reversed_kernel<__nv_bfloat16><<<grid_for(rows * H), 256, 0, st>>>(
            static_cast<__nv_bfloat16 *>(y), static_cast<const __nv_bfloat16 *>(yr), B, L, H);
    else if (H % 4 == 0)
        add_reversed_kernel<float4><<<grid_for(rows * (H / 4)), 256, 0, st>>>(
            static_cast<float4 *>(y), static_cast<const float4 *>(yr), B, L, H / 4);
    else
        add_reversed_kernel<float><<<grid_for(rows * H), 256, 0, st>>>(static_cast<float *>(y),
                                                                      static_cast<const float *>(yr), B, L, H);
    return cudaGetLastError();
}

}  // namespace s5
