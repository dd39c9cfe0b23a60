// The per-mode factors are computed in float-float arithmetic (s5_ff.cuh:
// about 48 significant bits from FP32 instructions) and rounded once to
// float, so they agree with a float64 evaluation to within one rounding.
// The phase Im(lambda)*Delta reaches tens of radians, so it needs more than
// float precision before its sine and cosine are taken; GB300's float64 pipe
// is too slow for the latency-bound chain (exp, then sin/cos, then a divide)
// that each mode is.  A complex expm1 keeps small |z| exact:
//   e^z - 1 = (e^x cos y - 1) + i e^x sin y,
//   e^x cos y - 1 = expm1(x) - vers(y) - expm1(x) vers(y),  vers = 1 - cos,
// with expm1 and vers from their own series (no cancellation near 0); the
// quotient by lambda then tends to Delta as z -> 0 without a separate branch.
#include "s5_internal.cuh"
#include "s5_ff.cuh"

namespace s5 {

namespace {

// Options of s5_discretize_ex, as float-float values.
struct DiscOpts {
    int method;          // 0 zero-order hold, 1 bilinear
    int clip_on;         // clip_eigs: Re(lambda) <- min(Re(lambda), clip)
    ff::F2 clip, scale;  // clip threshold; Delta multiplier (1 when not rescaling)
};

// lambda_bar (rounded) and the gain g = (lambda_bar - 1)/lambda (ZOH) or
// Delta/(1 - Delta lambda/2) (bilinear), g in float-float.
__device__ __forceinline__ void mode_factors(float2 l, float log_dt, const DiscOpts &o, float2 &lbar,
                                             ff::F2 &g_re, ff::F2 &g_im) {
    using namespace ff;
    F2 lr = make(l.x);
    const float li = l.y;
    // Re(lambda) > clip, compared exactly in float-float
    if (o.clip_on && (l.x > o.clip.hi || (l.x == o.clip.hi && o.clip.lo < 0.f))) lr = o.clip;
    F2 dt, unused;
    exp_expm1(make(log_dt), dt, unused);
    dt = mul(dt, o.scale);
    const F2 zr = mul(lr, dt), zi = mul(dt, li);
    if (o.method == 1) {
        // lambda_bar = (1 + z/2) / (1 - z/2), g = Delta / (1 - z/2)
        const F2 hr = mul(zr, 0.5f), hi = mul(zi, 0.5f);
        const F2 nr = add(make(1.f), hr), dr = sub(make(1.f), hr);
        // 1/(dr - i hi) = (dr + i hi) / (dr^2 + hi^2)
        const F2 inv = recip(add(mul(dr, dr), mul(hi, hi)));
        lbar = make_float2(to_float(mul(sub(mul(nr, dr), mul(hi, hi)), inv)),
                           to_float(mul(add(mul(hi, dr), mul(nr, hi)), inv)));
        g_re = mul(mul(dt, dr), inv);
        g_im = mul(mul(dt, hi), inv);
        return;
    }
    F2 ez, em1, sn, cs, vs;
    exp_expm1(zr, ez, em1);
    sincos_vers(zi, sn, cs, vs);
    lbar = make_float2(to_float(mul(ez, cs)), to_float(mul(ez, sn)));
    if (lr.hi == 0.f && li == 0.f) {
        // the removable singularity: (e^z - 1)/lambda -> Delta
        g_re = dt;
        g_im = make(0.f);
        return;
    }
    const F2 A = sub(sub(em1, vs), mul(em1, vs));   // Re(e^z - 1)
    const F2 Bm = mul(ez, sn);                       // Im(e^z - 1)
    // (A + iB) / (lr + i li) = ((A lr + B li) + i (B lr - A li)) / |lambda|^2
    const F2 inv = recip(add(mul(lr, lr), two_prod(li, li)));
    g_re = mul(add(mul(A, lr), mul(Bm, li)), inv);
    g_im = mul(sub(mul(Bm, lr), mul(A, li)), inv);
}

}  // namespace

// One block per mode; every thread computes the mode's factors (the same
// values in every lane: no barrier, no shared memory) and then scales its
// slice of the B_tilde row:  B_bar = g * B_tilde, formed in float-float and
// rounded once.
//
// Options (applied before the factors above):
//   clip_on        clip_eigs: Re(lambda) <- min(Re(lambda), clip_re)
//                  (wikillm "Paper vs code": the official value is -1e-4);
//   scale          sampling-rate rescaling, Delta <- Delta * dt_scale with
//                  dt_scale = old rate / new rate (review "Sampling intervals
//                  carry physical meaning"; summary section 6.2);
//   method 1       bilinear transform instead of the zero-order hold (review
//                  "Discretization controls both retention and input gain";
//                  the S4 page, "Discretize"): for a diagonal mode
//                  lambda_bar = (1 + Delta lambda/2) / (1 - Delta lambda/2) and
//                  gain = Delta / (1 - Delta lambda/2).
__global__ void discretize_kernel(const float2 *__restrict__ lambda, const float *__restrict__ log_dt,
                                  const float2 *__restrict__ b_tilde, int P, int H,
                                  float2 *__restrict__ lambda_bar, float2 *__restrict__ b_bar,
                                  const DiscOpts opts) {
    const int p = blockIdx.x;
    // the kernel that consumes Lambda_bar and B_bar may be scheduled now; it
    // waits for this one to complete before reading them
    griddep_launch_dependents();
    // Launched programmatically, this kernel may start while the kernel
    // before it still runs: it reads only its inputs (lambda, log_dt,
    // B_tilde, which the kernels of this library never write) before the
    // wait below, and writes Lambda_bar and B_bar, which that kernel may
    // still be reading, only after it.
    const float2 *src = b_tilde + (size_t)p * H;
    // this thread's first B_tilde element, fetched now so that its latency
    // overlaps the arithmetic below
    const float2 bt0 = (int)threadIdx.x < H ? src[threadIdx.x] : make_float2(0.f, 0.f);
    float2 lb;
    ff::F2 g_re, g_im;
    mode_factors(lambda[p], log_dt[p], opts, lb, g_re, g_im);
    griddep_wait();
    if (threadIdx.x == 0) lambda_bar[p] = lb;
    float2 *dst = b_bar + (size_t)p * H;
    for (int h = threadIdx.x; h < H; h += blockDim.x) {
        const float2 bt = h == (int)threadIdx.x ? bt0 : src[h];
        using namespace ff;
        const F2 re = sub(mul(g_re, bt.x), mul(g_im, bt.y));
        const F2 im = add(mul(g_re, bt.y), mul(g_im, bt.x));
        dst[h] = make_float2(to_float(re), to_float(im));
    }
}

// Per-mode constants of the irregular-sampling path (see ModeConst).
__global__ void mode_consts_kernel(const float2 *__restrict__ lambda, const float *__restrict__ log_dt,
                                   int P, ModeConst *__restrict__ out) {
    const int p = blockIdx.x * blockDim.x + threadIdx.x;
    if (p >= P) return;
    float2 l = lambda[p];
    double lr = l.x, li = l.y;
    double dt = exp((double)log_dt[p]);
    double om = li * dt;
    ModeConst m;
    m.om_hi = (float)om;
    m.om_lo = (float)(om - (double)m.om_hi);
    m.rho = (float)(lr * dt);
    m.dt = (float)dt;
    double den = lr * lr + li * li;
    m.inv_re = den > 0 ? (float)(lr / den) : 0.f;
    m.inv_im = den > 0 ? (float)(-li / den) : 0.f;
    m.zabs = (float)(sqrt(den) * dt);
    m.pad = 0.f;
    out[p] = m;
}

cudaError_t launch_discretize(const float2 *lambda, const float *log_dt, const float2 *b_tilde,
                              int P, int H, float2 *lambda_bar, float2 *b_bar, cudaStream_t st, int method,
                              double clip_re, double dt_scale) {
    DiscOpts o;
    o.method = method;
    o.clip_on = clip_re != 0.0;
    o.clip.hi = (float)clip_re;
    o.clip.lo = (float)(clip_re - (double)o.clip.hi);
    o.scale.hi = (float)dt_scale;
    o.scale.lo = (float)(dt_scale - (double)o.scale.hi);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)P);
    cfg.blockDim = dim3(H >= 256 ? 256 : (unsigned)((H + 31) / 32 * 32));
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    set_programmatic(attr[0]);
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, discretize_kernel, lambda, log_dt, b_tilde, P, H, lambda_bar, b_bar, o);
}

cudaError_t launch_mode_consts(const float2 *lambda, const float *log_dt, int P, ModeConst *out,
                               cudaStream_t st) {
    // a few modes per block so that the float64 work spreads over many SMs
    const int threads = 32;
    mode_consts_kernel<<<(P + threads - 1) / threads, threads, 0, st>>>(lambda, log_dt, P, out);
    return cudaGetLastError();
}

}  // namespace s5
