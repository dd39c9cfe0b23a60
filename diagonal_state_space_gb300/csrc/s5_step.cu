// s5_step.cu -- the streaming step and the helpers of the bidirectional layer.
//
// Streaming step (review "S5: Simplified State Space Layers for Sequence
// Modeling", "Associative scans preserve the recurrence": streaming inference
// keeps just the current state per layer; summary "SIMPLIFIED STATE SPACE
// LAYERS ...", App. C.1, online generation):
//   x <- lambda_bar * x + B_bar u,   y = 2 Re(C~ x) + D u.
// One block per sequence: u and the new state are staged in shared memory; a
// warp per mode forms (B_bar u)_p with lanes striding over the features
// (coalesced rows of B_bar), then a warp per feature forms the readout with
// lanes striding over the modes.
//
// Bidirectional layer ("Simplified State Space Layers for Sequence Modeling",
// "Paper vs code": a forward and a backward scan, C~ with 2P columns): the
// helpers split C~ into its two [H,P] halves, reverse sequences in time and add
// a time-reversed result into y.
#include <cuda_bf16.h>

#include "s5_internal.cuh"

namespace s5 {
namespace {

constexpr int STEP_THREADS = 256;

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__global__ void step_kernel(const float2 *__restrict__ lambda_bar, const float2 *__restrict__ b_bar,
                            const float2 *__restrict__ c_tilde, const float *__restrict__ d,
                            float2 *__restrict__ x, const float *__restrict__ u, float *__restrict__ y, int H,
                            int P) {
    extern __shared__ float2 sm_step[];
    float2 *sx = sm_step;                                // [P]
    float *su = reinterpret_cast<float *>(sm_step + P);  // [H]
    const int b = blockIdx.x, lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int nwarps = blockDim.x >> 5;
    const float *ub = u + (size_t)b * H;
    for (int h = threadIdx.x; h < H; h += blockDim.x) su[h] = ub[h];
    __syncthreads();
    for (int p = warp; p < P; p += nwarps) {
        const float2 *row = b_bar + (size_t)p * H;
        float re = 0.f, im = 0.f;
        for (int h = lane; h < H; h += 32) {
            const float2 w = row[h];
            re = fmaf(w.x, su[h], re);
            im = fmaf(w.y, su[h], im);
        }
        re = warp_sum(re);
        im = warp_sum(im);
        if (lane == 0) {
            const float2 lb = lambda_bar[p], xo = x[(size_t)b * P + p];
            const float2 xn = make_float2(fmaf(lb.x, xo.x, fmaf(-lb.y, xo.y, re)), fmaf(lb.x, xo.y, fmaf(lb.y, xo.x, im)));
            x[(size_t)b * P + p] = xn;
            sx[p] = xn;
        }
    }
    __syncthreads();
    for (int h = warp; h < H; h += nwarps) {
        const float2 *row = c_tilde + (size_t)h * P;
        float acc = 0.f;
        for (int p = lane; p < P; p += 32) {
            const float2 c = row[p], xv = sx[p];
            acc = fmaf(c.x, xv.x, fmaf(-c.y, xv.y, acc));
        }
        acc = warp_sum(acc);
        if (lane == 0) y[(size_t)b * H + h] = fmaf(d[h], su[h], 2.f * acc);
    }
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

size_t step_smem_bytes(int H, int P) { return sizeof(float2) * (size_t)P + sizeof(float) * (size_t)H; }

cudaError_t launch_step(const float2 *lambda_bar, const float2 *b_bar, const float2 *c_tilde, const float *d,
                        float2 *x, const float *u, float *y, int B, int H, int P, cudaStream_t st) {
    step_kernel<<<B, STEP_THREADS, step_smem_bytes(H, P), st>>>(lambda_bar, b_bar, c_tilde, d, x, u, y, H, P);
    return cudaGetLastError();
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
