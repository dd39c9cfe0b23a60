// s5_internal.cuh -- pieces shared by the kernels of libs5.so: workspace
// layout, latched device status, bounded flag waits and small complex helpers.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "../../include/s5.h"

namespace s5 {

// Row-major C[M][N] (fp32) = op(A) op(B) with bf16 operands: A is [M][K], or
// [K][M] with ta; B is [K][N], or [N][K] with tb; row pitches in elements
// (s5_gemm.cu).  Asynchronous on st.
cudaError_t gemm_bf16(cudaStream_t st, bool ta, bool tb, int M, int N, int K, const void *A, long long lda,
                      const void *B, long long ldb, float *C, long long ldc);
// Reads and clears the flag set when a wait inside the GEMM kernel ran out
// (1), 0 if none, -1 if the flag could not be read.
int gemm_fault_take();

// Records a CUDA error as the text s5_last_cuda_error() returns and gives
// S5_ERR_CUDA (defined with the entry points in s5_api.cu).
s5_status cuda_failure(cudaError_t e);

// ---------------------------------------------------------------------------
// Workspace.  The chunked scan publishes, per tile of T tokens of one
// sequence, the tile's aggregate map (A, E) = (product of a_k, end state from a
// zero start) and then its inclusive end state.  Layout (each region 256-byte
// aligned):
//   header (256 B) | flags [ntiles] u32 | agg [ntiles][P] float4 |
//   incl [ntiles][P] 16 bytes (the CUDA-core path uses the first 8 bytes of
//   each, as float2; the tensor-core path whole, as carry records) |
//   mode constants [P] ModeConst |
//   operand images [8*P*H bytes] (bf16 weights of the tensor-core path)
// Flags carry a launch epoch in their upper 30 bits so that a workspace needs
// no clearing between calls: the last CTA of every launch bumps the epoch and
// resets the tile counters.
// ---------------------------------------------------------------------------
struct WsHeader {
    unsigned int status;        // first device-side s5_status latched (0 = none)
    unsigned int tile_counter;  // dynamic, in-order tile claiming
    unsigned int done_counter;  // CTAs finished in this launch
    unsigned int epoch;         // launch generation stamped into the flags
    unsigned int drop_publish;  // diagnostics: tile+1 whose flags are never published
    unsigned int wait_limit_us; // diagnostics: carry-wait limit (0 = 1 s)
    unsigned int timeout_tile;  // diagnostics: tile+1 of the first wait that gave up
    unsigned int reserved[57];
};
static_assert(sizeof(WsHeader) == 256, "header is 256 bytes");

// Per-mode constants of the irregular-sampling path, computed in float64.
struct ModeConst {
    float om_hi, om_lo;   // omega = Im(lambda)*Delta as a float pair (hi + lo)
    float rho;            // Re(lambda)*Delta
    float dt;             // Delta
    float inv_re, inv_im; // 1/lambda
    float zabs;           // |lambda|*Delta
    float pad;
};
static_assert(sizeof(ModeConst) == 32, "ModeConst is 32 bytes");

constexpr unsigned FLAG_AGG = 1u, FLAG_INCL = 2u;

__host__ __device__ inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

struct WsLayout {
    WsHeader *hdr;
    unsigned int *flags;
    float4 *agg;
    float2 *incl;     // [ntiles][P] float2 (CUDA-core path)
    float4 *carry;    // the same region as [ntiles][P] float4 (tensor-core path)
    ModeConst *modes;
    unsigned char *wimg;
};

// Bytes of the bf16 operand images: B_bar split into 2P rows of H, and C' as
// H rows of 2P, 2 bytes each.
__host__ __device__ inline size_t wimg_bytes(int P, int H) { return (size_t)8 * P * H; }

__host__ __device__ inline size_t ws_bytes(long long ntiles, int P, int H) {
    size_t s = 256;
    s += align256(sizeof(unsigned int) * (size_t)ntiles);
    s += align256(sizeof(float4) * (size_t)ntiles * P);
    s += align256(sizeof(float4) * (size_t)ntiles * P);
    s += align256(sizeof(ModeConst) * (size_t)P);
    s += 1024 + wimg_bytes(P, H);   // images start 1024-byte aligned
    return s;
}

inline WsLayout ws_layout(void *base, long long ntiles, int P) {
    char *p = static_cast<char *>(base);
    WsLayout w;
    w.hdr = reinterpret_cast<WsHeader *>(p);
    p += 256;
    w.flags = reinterpret_cast<unsigned int *>(p);
    p += align256(sizeof(unsigned int) * (size_t)ntiles);
    w.agg = reinterpret_cast<float4 *>(p);
    p += align256(sizeof(float4) * (size_t)ntiles * P);
    w.incl = reinterpret_cast<float2 *>(p);
    w.carry = reinterpret_cast<float4 *>(p);
    p += align256(sizeof(float4) * (size_t)ntiles * P);
    w.modes = reinterpret_cast<ModeConst *>(p);
    p += align256(sizeof(ModeConst) * (size_t)P);
    // 1024-byte alignment keeps the swizzle pattern of the images intact
    p = reinterpret_cast<char *>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
    w.wimg = reinterpret_cast<unsigned char *>(p);
    return w;
}

// ---------------------------------------------------------------------------
// Device helpers.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void latch_status(WsHeader *h, unsigned code) {
    atomicCAS(&h->status, 0u, code);
}

// Programmatic dependent launch.  A kernel launched with the programmatic
// stream-serialisation attribute may be scheduled while the kernel before it
// in the stream is still running; griddep_wait() returns once that kernel
// has completed and its writes are visible, so every read or write of memory
// the previous kernel may touch comes after it.  In a kernel launched without
// the attribute it returns at once.  griddep_launch_dependents() lets the
// next such kernel be scheduled before this one ends.
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

inline void set_programmatic(cudaLaunchAttribute &a) {
    a.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    a.val.programmaticStreamSerializationAllowed = 1;
}

__device__ __forceinline__ unsigned ld_acquire(const unsigned int *p) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void st_release(unsigned int *p, unsigned v) {
    asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ unsigned long long global_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Waits (bounded) until flag *f carries this launch's epoch and a non-zero
// state; returns FLAG_AGG / FLAG_INCL, or 0 if the wait gave up (the status
// S5_ERR_TIMEOUT is then latched and the caller treats the tile as holding a
// zero inclusive state, so that every later tile still completes).
__device__ inline unsigned wait_flag(WsHeader *hdr, const unsigned int *f, unsigned epoch,
                                     unsigned long long limit_ns, unsigned tile) {
    unsigned long long t0 = 0;
    unsigned backoff = 32;
    for (unsigned iter = 0;; ++iter) {
        unsigned v = ld_acquire(f);
        if ((v >> 2) == epoch && (v & 3u) != 0) return v & 3u;
        if (iter == 0) t0 = global_ns();
        else if (global_ns() - t0 > limit_ns) {
            latch_status(hdr, S5_ERR_TIMEOUT);
            atomicCAS(&hdr->timeout_tile, 0u, tile + 1);
            return 0;
        }
        __nanosleep(backoff);
        if (backoff < 128) backoff <<= 1;
    }
}

__device__ __forceinline__ float2 cmul(float2 a, float2 b) {
    return make_float2(fmaf(a.x, b.x, -a.y * b.y), fmaf(a.x, b.y, a.y * b.x));
}
// a*b + c
__device__ __forceinline__ float2 cfma(float2 a, float2 b, float2 c) {
    return make_float2(fmaf(a.x, b.x, fmaf(-a.y, b.y, c.x)), fmaf(a.x, b.y, fmaf(a.y, b.x, c.y)));
}

template <typename T> __device__ __forceinline__ float load_elem(const T *p);
template <> __device__ __forceinline__ float load_elem<float>(const float *p) { return __ldg(p); }
template <> __device__ __forceinline__ float load_elem<__nv_bfloat16>(const __nv_bfloat16 *p) {
    return __bfloat162float(*p);
}
template <typename T> __device__ __forceinline__ void store_elem(T *p, float v);
template <> __device__ __forceinline__ void store_elem<float>(float *p, float v) { *p = v; }
template <> __device__ __forceinline__ void store_elem<__nv_bfloat16>(__nv_bfloat16 *p, float v) {
    *p = __float2bfloat16_rn(v);
}

}  // namespace s5
