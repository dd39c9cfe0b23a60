// s5_api.cu -- the C entry points of libs5.so: argument checks, kernel
// selection and launch.  Every numeric step runs in the kernels; this file
// only validates, chooses a kernel and queues it on the caller's stream.
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "s5_simt.cuh"
#include "s5_tc.cuh"

namespace s5 {
cudaError_t launch_discretize(const float2 *, const float *, const float2 *, int, int, float2 *,
                              float2 *, cudaStream_t, int method = 0, double clip_re = 0.0, double dt_scale = 1.0);
cudaError_t launch_mode_consts(const float2 *, const float *, int, ModeConst *, cudaStream_t);
size_t step_smem_bytes(int H, int P);
cudaError_t launch_step(const float2 *, const float2 *, const float2 *, const float *, float2 *, const float *,
                        float *, int B, int H, int P, cudaStream_t);
cudaError_t launch_split_c(const float2 *, int H, int P, float2 *, float2 *, cudaStream_t);
cudaError_t launch_reverse_time(const void *, void *, int B, int L, int H, int elem_bytes, cudaStream_t);
cudaError_t launch_add_reversed(void *, const void *, int B, int L, int H, bool bf16, cudaStream_t);
}  // namespace s5

namespace {

thread_local char g_cuda_err[256] = "";

s5_status cuda_fail(cudaError_t e) {
    std::snprintf(g_cuda_err, sizeof(g_cuda_err), "%s: %s", cudaGetErrorName(e), cudaGetErrorString(e));
    return S5_ERR_CUDA;
}

bool aligned16(const void *p) { return (reinterpret_cast<std::uintptr_t>(p) & 15u) == 0; }

int num_sms_current() {
    static std::mutex mu;
    static int cache[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    std::lock_guard<std::mutex> lk(mu);
    if (!cache[dev]) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
        cache[dev] = n;
    }
    return cache[dev];
}

bool dtype_ok(s5_dtype d) { return d == S5_F32 || d == S5_BF16; }

long long ceil_div(long long a, long long b) { return (a + b - 1) / b; }

// Smallest tile (tokens) any forward kernel may pick for these sizes; the
// workspace is sized for it.
int min_tile_tokens(int H, int P) {
    int t0 = s5::simt_tile_tokens(H, P, false);
    int t1 = s5::simt_tile_tokens(H, P, true);
    int t = t0 == 0 ? t1 : (t1 == 0 ? t0 : (t0 < t1 ? t0 : t1));
    if (s5::tc_supported(H, P, true, true, true) && (t == 0 || s5::TC_TILE_TOKENS < t))
        t = s5::TC_TILE_TOKENS;
    return t;
}

// Shared checks of the two forward entry points.
s5_status check_forward(const void *c_tilde, const void *d, const void *u, s5_dtype u_dtype,
                        const void *y, s5_dtype y_dtype, s5_dtype proj_dtype, int B, int L, int H,
                        int P, const void *x0, const void *x_last, const void *ws,
                        size_t ws_bytes) {
    if (B < 0 || L < 0 || H < 1 || P < 1) return S5_ERR_INVALID_ARGUMENT;
    if (!dtype_ok(u_dtype) || !dtype_ok(y_dtype) || !dtype_ok(proj_dtype))
        return S5_ERR_INVALID_ARGUMENT;
    if (!c_tilde || !d || !aligned16(c_tilde) || !aligned16(d)) return S5_ERR_INVALID_ARGUMENT;
    if (x0 && !aligned16(x0)) return S5_ERR_INVALID_ARGUMENT;
    if (x_last && !aligned16(x_last)) return S5_ERR_INVALID_ARGUMENT;
    if ((long long)B * L == 0) return S5_OK;
    if (!u || !y || !aligned16(u) || !aligned16(y)) return S5_ERR_INVALID_ARGUMENT;
    if (!ws || !aligned16(ws)) return S5_ERR_INVALID_ARGUMENT;
    if (ws_bytes < s5_workspace_size(B, L, H, P)) return S5_ERR_INVALID_ARGUMENT;
    return S5_OK;
}

// B = 0 or L = 0: nothing to compute; x_last (if any) receives x0 or zeros.
s5_status empty_forward(int B, int P, const float *x0, float *x_last, cudaStream_t st) {
    if (!x_last || B == 0) return S5_OK;
    size_t bytes = sizeof(float) * 2 * (size_t)B * P;
    cudaError_t e = x0 ? cudaMemcpyAsync(x_last, x0, bytes, cudaMemcpyDeviceToDevice, st)
                       : cudaMemsetAsync(x_last, 0, bytes, st);
    return e == cudaSuccess ? S5_OK : cuda_fail(e);
}

s5_status run_simt(const float2 *lambda_bar, const float2 *w, const float2 *c_tilde, const float *d,
                   const float *g, const void *u, s5_dtype u_dtype, void *y, s5_dtype y_dtype,
                   int B, int L, int H, int P, const float *x0, float *x_last, void *workspace,
                   bool varying, cudaStream_t st) {
    const int T = s5::simt_tile_tokens(H, P, varying);
    if (T == 0) return S5_ERR_UNSUPPORTED;
    const int sms = num_sms_current();
    if (sms == 0) return cuda_fail(cudaGetLastError());
    const long long nchunks = ceil_div(L, T);
    const long long ntiles = nchunks * B;
    if (ntiles >= (1ll << 31)) return S5_ERR_UNSUPPORTED;
    s5::SimtArgs a;
    a.lambda_bar = lambda_bar;
    a.w = w;
    a.c_tilde = c_tilde;
    a.d = d;
    a.u = u;
    a.y = y;
    a.x0 = reinterpret_cast<const float2 *>(x0);
    a.x_last = reinterpret_cast<float2 *>(x_last);
    a.g = g;
    a.B = B;
    a.L = L;
    a.H = H;
    a.P = P;
    a.T = T;
    a.nchunks = (int)nchunks;
    a.nseg = s5::simt_nseg(P);
    a.ntiles = ntiles;
    a.ws = s5::ws_layout(workspace, ntiles, P);
    cudaError_t e = s5::launch_forward_simt(a, u_dtype == S5_BF16, y_dtype == S5_BF16, varying,
                                            st, sms);
    return e == cudaSuccess ? S5_OK : cuda_fail(e);
}

// Tensor-core path: bf16 operands, fp32 accumulation, complex fp32 scan.
s5_status run_tc(const float2 *lambda_bar, const float2 *b_bar, const float2 *c_tilde,
                 const float *d, const void *u, void *y, int B, int L, int H, int P,
                 const float *x0, float *x_last, void *workspace, cudaStream_t st) {
    const int sms = num_sms_current();
    if (sms == 0) return cuda_fail(cudaGetLastError());
    const long long nchunks = ceil_div(L, s5::TC_TILE_TOKENS);
    const long long ntiles = nchunks * B;
    if (ntiles >= (1ll << 31)) return S5_ERR_UNSUPPORTED;
    s5::TcArgs a;
    a.lambda_bar = lambda_bar;
    a.b_bar = b_bar;
    a.c_tilde = c_tilde;
    a.d = d;
    a.y = y;
    a.x0 = reinterpret_cast<const float2 *>(x0);
    a.x_last = reinterpret_cast<float2 *>(x_last);
    a.B = B;
    a.L = L;
    a.nchunks = (int)nchunks;
    a.ntiles = (int)ntiles;
    a.ws = s5::ws_layout(workspace, ntiles, P);
    (void)H;
    cudaError_t e = s5::launch_forward_tc(a, u, st, sms);
    return e == cudaSuccess ? S5_OK : cuda_fail(e);
}

// The backward scan of the bidirectional layer on the tensor-core path: adds
// 2 Re(c_tilde_b xb_k) into y, scanning each sequence from its end.
s5_status run_tc_backward_add(const float2 *lambda_bar, const float2 *b_bar, const float2 *c_tilde_b,
                              const void *u, void *y, int B, int L, int P, void *workspace, cudaStream_t st) {
    const int sms = num_sms_current();
    if (sms == 0) return cuda_fail(cudaGetLastError());
    const long long nchunks = ceil_div(L, s5::TC_TILE_TOKENS);
    const long long ntiles = nchunks * B;
    if (ntiles >= (1ll << 31)) return S5_ERR_UNSUPPORTED;
    s5::TcArgs a;
    a.lambda_bar = lambda_bar;
    a.b_bar = b_bar;
    a.c_tilde = c_tilde_b;
    a.d = nullptr;
    a.y = y;
    a.x0 = nullptr;
    a.x_last = nullptr;
    a.B = B;
    a.L = L;
    a.nchunks = (int)nchunks;
    a.ntiles = (int)ntiles;
    a.ws = s5::ws_layout(workspace, ntiles, P);
    cudaError_t e = s5::launch_backward_add_tc(a, u, st, sms);
    return e == cudaSuccess ? S5_OK : cuda_fail(e);
}

}  // namespace

namespace s5 {
s5_status cuda_failure(cudaError_t e) { return cuda_fail(e); }
}  // namespace s5

extern "C" {

const char *s5_status_string(s5_status s) {
    switch (s) {
    case S5_OK: return "ok";
    case S5_ERR_INVALID_ARGUMENT: return "invalid argument";
    case S5_ERR_UNSUPPORTED: return "unsupported sizes or types";
    case S5_ERR_CUDA: return "CUDA error";
    case S5_ERR_TIMEOUT: return "carry wait timed out";
    case S5_ERR_NONFINITE: return "non-finite or negative interval";
    }
    return "unknown status";
}

const char *s5_last_cuda_error(void) { return g_cuda_err; }

size_t s5_workspace_size(int B, int L, int H, int P) {
    if (B < 0 || L < 0 || H < 1 || P < 1) return 0;
    const int T = min_tile_tokens(H, P);
    if (T == 0) return 0;
    const long long ntiles = (long long)B * ceil_div(L, T);
    return s5::ws_bytes(ntiles, P, H);
}

s5_status s5_discretize(const float *lambda, const float *log_dt, const float *b_tilde, int P,
                        int H, float *lambda_bar, float *b_bar, s5_stream_t stream) {
    if (P < 1 || H < 1) return S5_ERR_INVALID_ARGUMENT;
    const void *ptrs[] = {lambda, log_dt, b_tilde, lambda_bar, b_bar};
    for (const void *p : ptrs)
        if (!p || !aligned16(p)) return S5_ERR_INVALID_ARGUMENT;
    cudaError_t e = s5::launch_discretize(
        reinterpret_cast<const float2 *>(lambda), log_dt, reinterpret_cast<const float2 *>(b_tilde),
        P, H, reinterpret_cast<float2 *>(lambda_bar), reinterpret_cast<float2 *>(b_bar),
        reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? S5_OK : cuda_fail(e);
}

s5_status s5_discretize_ex(const float *lambda, const float *log_dt, const float *b_tilde, int P, int H,
                           s5_discretization method, float clip_re, float dt_scale, float *lambda_bar,
                           float *b_bar, s5_stream_t stream) {
    if (P < 1 || H < 1) return S5_ERR_INVALID_ARGUMENT;
    if (method != S5_ZOH && method != S5_BILINEAR) return S5_ERR_INVALID_ARGUMENT;
    if (!(dt_scale > 0.f) || !(clip_re <= 0.f)) return S5_ERR_INVALID_ARGUMENT;   // also rejects NaN
    const void *ptrs[] = {lambda, log_dt, b_tilde, lambda_bar, b_bar};
    for (const void *p : ptrs)
        if (!p || !aligned16(p)) return S5_ERR_INVALID_ARGUMENT;
    cudaError_t e = s5::launch_discretize(
        reinterpret_cast<const float2 *>(lambda), log_dt, reinterpret_cast<const float2 *>(b_tilde),
        P, H, reinterpret_cast<float2 *>(lambda_bar), reinterpret_cast<float2 *>(b_bar),
        reinterpret_cast<cudaStream_t>(stream), (int)method, (double)clip_re, (double)dt_scale);
    return e == cudaSuccess ? S5_OK : cuda_fail(e);
}

s5_status s5_forward(const float *lambda_bar, const float *b_bar, const float *c_tilde,
                     const float *d, const void *u, s5_dtype u_dtype, void *y, s5_dtype y_dtype,
                     s5_dtype proj_dtype, int B, int L, int H, int P, const float *x0,
                     float *x_last, void *workspace, size_t workspace_bytes, s5_stream_t stream) {
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (!lambda_bar || !b_bar || !aligned16(lambda_bar) || !aligned16(b_bar))
        return S5_ERR_INVALID_ARGUMENT;
    s5_status s = check_forward(c_tilde, d, u, u_dtype, y, y_dtype, proj_dtype, B, L, H, P, x0,
                                x_last, workspace, workspace_bytes);
    if (s != S5_OK) return s;
    if ((long long)B * L == 0) return empty_forward(B, P, x0, x_last, st);
    if (s5::tc_supported(H, P, u_dtype == S5_BF16, y_dtype == S5_BF16, proj_dtype == S5_BF16))
        return run_tc(reinterpret_cast<const float2 *>(lambda_bar),
                      reinterpret_cast<const float2 *>(b_bar),
                      reinterpret_cast<const float2 *>(c_tilde), d, u, y, B, L, H, P, x0, x_last,
                      workspace, st);
    return run_simt(reinterpret_cast<const float2 *>(lambda_bar),
                    reinterpret_cast<const float2 *>(b_bar),
                    reinterpret_cast<const float2 *>(c_tilde), d, nullptr, u, u_dtype, y, y_dtype,
                    B, L, H, P, x0, x_last, workspace, false, st);
}

s5_status s5_forward_varying_dt(const float *lambda, const float *log_dt, const float *b_tilde,
                                const float *c_tilde, const float *d, const float *dt_scale,
                                const void *u, s5_dtype u_dtype, void *y, s5_dtype y_dtype,
                                s5_dtype proj_dtype, int B, int L, int H, int P,
                                const float *x0, float *x_last, void *workspace,
                                size_t workspace_bytes, s5_stream_t stream) {
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (!lambda || !log_dt || !b_tilde || !aligned16(lambda) || !aligned16(log_dt) ||
        !aligned16(b_tilde))
        return S5_ERR_INVALID_ARGUMENT;
    s5_status s = check_forward(c_tilde, d, u, u_dtype, y, y_dtype, proj_dtype, B, L, H, P, x0,
                                x_last, workspace, workspace_bytes);
    if (s != S5_OK) return s;
    if ((long long)B * L == 0) return empty_forward(B, P, x0, x_last, st);
    if (!dt_scale || !aligned16(dt_scale)) return S5_ERR_INVALID_ARGUMENT;
    const int T = s5::simt_tile_tokens(H, P, true);
    if (T == 0) return S5_ERR_UNSUPPORTED;
    const long long ntiles = (long long)B * ceil_div(L, T);
    s5::WsLayout ws = s5::ws_layout(workspace, ntiles, P);
    cudaError_t e = s5::launch_mode_consts(reinterpret_cast<const float2 *>(lambda), log_dt, P,
                                           ws.modes, st);
    if (e != cudaSuccess) return cuda_fail(e);
    return run_simt(nullptr, reinterpret_cast<const float2 *>(b_tilde),
                    reinterpret_cast<const float2 *>(c_tilde), d, dt_scale, u, u_dtype, y,
                    y_dtype, B, L, H, P, x0, x_last, workspace, true, st);
}

s5_status s5_step(const float *lambda_bar, const float *b_bar, const float *c_tilde, const float *d,
                  float *x, const float *u, float *y, int B, int H, int P, s5_stream_t stream) {
    if (B < 0 || H < 1 || P < 1) return S5_ERR_INVALID_ARGUMENT;
    const void *params[] = {lambda_bar, b_bar, c_tilde, d};
    for (const void *p : params)
        if (!p || !aligned16(p)) return S5_ERR_INVALID_ARGUMENT;
    if (B == 0) return S5_OK;
    const void *io[] = {x, u, y};
    for (const void *p : io)
        if (!p || !aligned16(p)) return S5_ERR_INVALID_ARGUMENT;
    if (s5::step_smem_bytes(H, P) > 200 * 1024) return S5_ERR_UNSUPPORTED;
    cudaError_t e = s5::launch_step(reinterpret_cast<const float2 *>(lambda_bar), reinterpret_cast<const float2 *>(b_bar),
                                    reinterpret_cast<const float2 *>(c_tilde), d, reinterpret_cast<float2 *>(x), u, y,
                                    B, H, P, reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? S5_OK : cuda_fail(e);
}

// Bidirectional workspace: the forward workspace, then (each 256-aligned) the
// time-reversed u, the backward scan's output, the two halves of c_tilde2 and
// a zero d.
struct BidiLayout {
    size_t fwd, ur, yr, cf, cb, d0, total;
};
static BidiLayout bidi_layout(int B, int L, int H, int P, s5_dtype u_dtype, s5_dtype y_dtype) {
    BidiLayout l{};
    auto al = [](size_t v) { return (v + 255) & ~(size_t)255; };
    const size_t nel = (size_t)B * L * H;
    l.fwd = al(s5_workspace_size(B, L, H, P));
    l.ur = l.fwd;
    l.yr = l.ur + al(nel * (u_dtype == S5_BF16 ? 2 : 4));
    l.cf = l.yr + al(nel * (y_dtype == S5_BF16 ? 2 : 4));
    l.cb = l.cf + al(sizeof(float) * 2 * (size_t)H * P);
    l.d0 = l.cb + al(sizeof(float) * 2 * (size_t)H * P);
    l.total = l.d0 + al(sizeof(float) * (size_t)H);
    return l;
}

size_t s5_bidirectional_workspace_size(int B, int L, int H, int P, s5_dtype u_dtype, s5_dtype y_dtype) {
    if (B < 0 || L < 0 || H < 1 || P < 1 || !dtype_ok(u_dtype) || !dtype_ok(y_dtype)) return 0;
    if (s5_workspace_size(B, L, H, P) == 0) return 0;
    return bidi_layout(B, L, H, P, u_dtype, y_dtype).total;
}

s5_status s5_forward_bidirectional(const float *lambda_bar, const float *b_bar, const float *c_tilde2,
                                   const float *d, const void *u, s5_dtype u_dtype, void *y,
                                   s5_dtype y_dtype, s5_dtype proj_dtype, int B, int L, int H, int P,
                                   void *workspace, size_t workspace_bytes, s5_stream_t stream) {
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (!lambda_bar || !b_bar || !aligned16(lambda_bar) || !aligned16(b_bar)) return S5_ERR_INVALID_ARGUMENT;
    if (B < 0 || L < 0 || H < 1 || P < 1) return S5_ERR_INVALID_ARGUMENT;
    if (!dtype_ok(u_dtype) || !dtype_ok(y_dtype) || !dtype_ok(proj_dtype)) return S5_ERR_INVALID_ARGUMENT;
    if (!c_tilde2 || !d || !aligned16(c_tilde2) || !aligned16(d)) return S5_ERR_INVALID_ARGUMENT;
    if ((long long)B * L == 0) return S5_OK;
    if (!u || !y || !aligned16(u) || !aligned16(y) || !workspace || !aligned16(workspace))
        return S5_ERR_INVALID_ARGUMENT;
    const size_t need = s5_bidirectional_workspace_size(B, L, H, P, u_dtype, y_dtype);
    if (need == 0 || (size_t)B * L * H >= (1ull << 31)) return S5_ERR_UNSUPPORTED;
    if (workspace_bytes < need) return S5_ERR_INVALID_ARGUMENT;
    const BidiLayout l = bidi_layout(B, L, H, P, u_dtype, y_dtype);
    char *w = static_cast<char *>(workspace);
    float2 *cf = reinterpret_cast<float2 *>(w + l.cf), *cb = reinterpret_cast<float2 *>(w + l.cb);
    float *d0 = reinterpret_cast<float *>(w + l.d0);
    cudaError_t e = s5::launch_split_c(reinterpret_cast<const float2 *>(c_tilde2), H, P, cf, cb, st);
    if (e != cudaSuccess) return cuda_fail(e);
    if (s5::tc_supported(H, P, u_dtype == S5_BF16, y_dtype == S5_BF16, proj_dtype == S5_BF16)) {
        // tensor-core path: the forward scan writes y, the backward scan adds
        // into it in place (no reversed copies)
        s5_status s = s5_forward(lambda_bar, b_bar, reinterpret_cast<const float *>(cf), d, u, u_dtype, y,
                                 y_dtype, proj_dtype, B, L, H, P, nullptr, nullptr, w, l.fwd, stream);
        if (s != S5_OK) return s;
        return run_tc_backward_add(reinterpret_cast<const float2 *>(lambda_bar),
                                   reinterpret_cast<const float2 *>(b_bar), cb, u, y, B, L, P, w, st);
    }
    e = cudaMemsetAsync(d0, 0, sizeof(float) * (size_t)H, st);
    if (e == cudaSuccess)
        e = s5::launch_reverse_time(u, w + l.ur, B, L, H, u_dtype == S5_BF16 ? 2 : 4, st);
    if (e != cudaSuccess) return cuda_fail(e);
    s5_status s = s5_forward(lambda_bar, b_bar, reinterpret_cast<const float *>(cf), d, u, u_dtype, y, y_dtype,
                             proj_dtype, B, L, H, P, nullptr, nullptr, w, l.fwd, stream);
    if (s != S5_OK) return s;
    s = s5_forward(lambda_bar, b_bar, reinterpret_cast<const float *>(cb), d0, w + l.ur, u_dtype, w + l.yr, y_dtype,
                   proj_dtype, B, L, H, P, nullptr, nullptr, w, l.fwd, stream);
    if (s != S5_OK) return s;
    e = s5::launch_add_reversed(y, w + l.yr, B, L, H, y_dtype == S5_BF16, st);
    return e == cudaSuccess ? S5_OK : cuda_fail(e);
}

s5_status s5_sync_status(void *workspace, s5_stream_t stream) {
    if (!workspace || !aligned16(workspace)) return S5_ERR_INVALID_ARGUMENT;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    s5::WsHeader *hdr = static_cast<s5::WsHeader *>(workspace);
    unsigned v = 0;
    cudaError_t e = cudaMemcpyAsync(&v, &hdr->status, sizeof(v), cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return cuda_fail(e);
    if (v != 0) {
        e = cudaMemsetAsync(&hdr->status, 0, sizeof(unsigned), st);
        if (e == cudaSuccess) e = cudaMemsetAsync(&hdr->timeout_tile, 0, sizeof(unsigned), st);
        if (e == cudaSuccess) e = cudaStreamSynchronize(st);
        if (e != cudaSuccess) return cuda_fail(e);
    }
    return static_cast<s5_status>(v);
}

}  // extern "C"
