// s5_tc.cuh -- arguments of the tensor-core forward kernel (s5_forward_tc.cu).
#pragma once
#include "s5_internal.cuh"

namespace s5 {

constexpr int TC_TILE_TOKENS = 64;

struct TcArgs {
    const float2 *lambda_bar;  // [P]
    const float2 *b_bar;       // [P][H]
    const float2 *c_tilde;     // [H][P]
    const float *d;            // [H]
    void *y;                   // [B][L][H] bf16
    const float2 *x0;          // [B][P] or null
    float2 *x_last;            // [B][P] or null
    const void *u;             // [B][L][H] bf16 (set by launch_forward_tc)
    int B, L, nchunks, ntiles;
    int W;                     // lanes per sequence (set by launch_forward_tc)
    WsLayout ws;               // aggregate records: values in ws.incl, flags in ws.flags
};

// The tensor-core kernel covers H = 128, P = 128 with bf16 u, y and projections.
bool tc_supported(int H, int P, bool u_bf16, bool y_bf16, bool proj_bf16);
// Lanes per sequence (W) and grid size (G) of the tensor-core launches.
void tc_grid(int B, int nchunks, int num_sms, int *W, int *G);
cudaError_t launch_forward_tc(const TcArgs &a, const void *u, cudaStream_t st, int num_sms);
// The backward scan of the bidirectional layer (a.c_tilde = the backward
// half of C~; a.d, a.x0, a.x_last unused): y += 2 Re(C~_b xb), with
// xb_k = lambda_bar xb_{k+1} + B_bar u_k over each sequence in reverse.
cudaError_t launch_backward_add_tc(const TcArgs &a, const void *u, cudaStream_t st, int num_sms);

}  // namespace s5
