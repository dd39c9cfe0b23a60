// s5_simt.cuh -- arguments of the CUDA-core forward kernel (s5_forward_simt.cu).
#pragma once
#include "s5_internal.cuh"

namespace s5 {

struct SimtArgs {
    const float2 *lambda_bar;  // [P] (time-invariant path)
    const float2 *w;           // B_bar, or B_tilde for irregular sampling, [P][H]
    const float2 *c_tilde;     // [H][P]
    const float *d;            // [H]
    const void *u;             // [B][L][H]
    void *y;                   // [B][L][H]
    const float2 *x0;          // [B][P] or null
    float2 *x_last;            // [B][P] or null
    const float *g;            // [B][L] gaps (irregular sampling)
    int B, L, H, P, T, nchunks, nseg;
    long long ntiles;
    WsLayout ws;
};

int simt_nseg(int P);
int simt_tile_tokens(int H, int P, bool varying);
cudaError_t launch_forward_simt(const SimtArgs &a, bool u_bf16, bool y_bf16, bool varying,
                                cudaStream_t st, int num_sms);

}  // namespace s5
