// Device code of the fused LM-head loss.
//
// Notation per active row r (logits z, target t, teacher u):
//   m_nt = max_{j!=t} z_j,  S_nt = sum_{j!=t} exp(z_j - m_nt),  lse_nt = m_nt + ln S_nt
//   NLL  = softplus(lse_nt - z_t),  lse = logaddexp(z_t, lse_nt),  p_j = exp(z_j - lse)
// torchtitan PR 5661 "fix softmax collapse with improved CE perf", commit
// message, "Numerics (TP > 1 only)": the target term is dropped before the sum
// (not subtracted after it) and the target gradient is p_t - 1 below p_t = 1/4,
// else -p_non_target.
#pragma once

#include <cuda_bf16.h>
#include <cstdint>

#include "ptx.cuh"

namespace lmloss {

constexpr float kLog2e = 1.4426950408889634f;

template <bool B>
struct BoolConst {
    static constexpr bool value = B;
};
constexpr long long kWaitLimitCycles = 4000000000LL;   // ~2 s at the top SM clock

// Device error codes (match lmloss_status).
enum : int { kErrBadTarget = 4, kErrBadSegment = 5, kErrRange = 6, kErrTimeout = 7 };

__device__ __forceinline__ void set_error(int* err, int code)
{
    atomicCAS(err, 0, code);
}

// ----------------------------------------------------------------- vectors
// One 16-byte vector of logits: 8 bf16 or 4 fp32.
template <bool BF16>
struct Vec;

template <>
struct Vec<true> {
    static constexpr int N = 8;
    static constexpr int ESZ = 2;
    __device__ static __forceinline__ void unpack(const uint4& q, float (&x)[8])
    {
        const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            x[2 * k] = __uint_as_float(w[k] << 16);
            x[2 * k + 1] = __uint_as_float(w[k] & 0xffff0000u);
        }
    }
    __device__ static __forceinline__ uint4 pack(const float (&g)[8])
    {
        uint32_t w[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            __nv_bfloat162 h = __floats2bfloat162_rn(g[2 * k], g[2 * k + 1]);
            w[k] = *reinterpret_cast<uint32_t*>(&h);
        }
        return make_uint4(w[0], w[1], w[2], w[3]);
    }
    // Running packed maximum; NaN lanes are skipped here and surface in the sum.
    __device__ static __forceinline__ uint32_t max_init() { return 0xff80ff80u; }  // (-inf, -inf)
    __device__ static __forceinline__ uint32_t max_acc(uint32_t acc, const uint4& q)
    {
        __nv_bfloat162 a = *reinterpret_cast<const __nv_bfloat162*>(&q.x);
        __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162*>(&q.y);
        __nv_bfloat162 c = *reinterpret_cast<const __nv_bfloat162*>(&q.z);
        __nv_bfloat162 d = *reinterpret_cast<const __nv_bfloat162*>(&q.w);
        __nv_bfloat162 m = __hmax2(__hmax2(a, b), __hmax2(c, d));
        __nv_bfloat162 r = __hmax2(m, *reinterpret_cast<__nv_bfloat162*>(&acc));
        return *reinterpret_cast<uint32_t*>(&r);
    }
    __device__ static __forceinline__ float max_final(uint32_t acc)
    {
        return fmaxf(__uint_as_float(acc << 16), __uint_as_float(acc & 0xffff0000u));
    }
    // Pair k (elements 2k, 2k+1) of a vector as packed fp32.
    __device__ static __forceinline__ uint64_t pair(const uint4& q, int k)
    {
        const uint32_t w = k == 0 ? q.x : (k == 1 ? q.y : (k == 2 ? q.z : q.w));
        return f2_pack(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
    }
    __device__ static __forceinline__ float load1(const void* base, int64_t idx)
    {
        const uint16_t b = reinterpret_cast<const uint16_t*>(base)[idx];
        return __uint_as_float(static_cast<uint32_t>(b) << 16);
    }
    __device__ static __forceinline__ void store1(void* base, int64_t idx, float v)
    {
        __nv_bfloat16 h = __float2bfloat16_rn(v);
        reinterpret_cast<__nv_bfloat16*>(base)[idx] = h;
    }
};

template <>
struct Vec<false> {
    static constexpr int N = 4;
    static constexpr int ESZ = 4;
    __device__ static __forceinline__ void unpack(const uint4& q, float (&x)[4])
    {
        x[0] = __uint_as_float(q.x);
        x[1] = __uint_as_float(q.y);
        x[2] = __uint_as_float(q.z);
        x[3] = __uint_as_float(q.w);
    }
    __device__ static __forceinline__ uint4 pack(const float (&g)[4])
    {
        return make_uint4(__float_as_uint(g[0]), __float_as_uint(g[1]), __float_as_uint(g[2]),
                          __float_as_uint(g[3]));
    }
    __device__ static __forceinline__ uint32_t max_init() { return 0xff800000u; }
    __device__ static __forceinline__ uint32_t max_acc(uint32_t acc, const uint4& q)
    {
        float m = fmaxf(fmaxf(__uint_as_float(q.x), __uint_as_float(q.y)),
                        fmaxf(__uint_as_float(q.z), __uint_as_float(q.w)));
        return __float_as_uint(fmaxf(m, __uint_as_float(acc)));
    }
    __device__ static __forceinline__ float max_final(uint32_t acc) { return __uint_as_float(acc); }
    __device__ static __forceinline__ uint64_t pair(const uint4& q, int k)
    {
        return k == 0 ? f2_pack(__uint_as_float(q.x), __uint_as_float(q.y))
                      : f2_pack(__uint_as_float(q.z), __uint_as_float(q.w));
    }
    __device__ static __forceinline__ float load1(const void* base, int64_t idx)
    {
        return reinterpret_cast<const float*>(base)[idx];
    }
    __device__ static __forceinline__ void store1(void* base, int64_t idx, float v)
    {
        reinterpret_cast<float*>(base)[idx] = v;
    }
};

// --------------------------------------------------------- softmax partials
// (m, s): s = sum 2^((x - m) L) over some set; m = -inf with s = 0 for the empty
// set.  L = log2 e gives s = sum exp(x - m); L = log2(e) / tau the same at the
// temperature tau.
__device__ __forceinline__ float rescale(float m, float M, float L = kLog2e)
{
    return (m == M) ? 1.0f : ex2((m - M) * L);
}

// ------------------------------------------------------------ parameters
struct Workspace {
    float* row_nll;      // [max_T]
    float* row_lse;      // [max_T]
    float* row_kl;       // [max_T]
    float* row_pol;      // [max_T] per-token GRPO loss
    float* row_tu;       // [max_T][2] teacher: Mu, ln Su (statistics pass with a teacher, for
                         //   GSPO's gradient pass)
    float* row_tt;       // [max_T][4] tau != 1: mr, rb, p^tau_t, 0 (likewise)
    int64_t* n_active;   // [1]
    int64_t* n_nonempty; // [1]
    double* gspo_sum;    // [1]  sum of L_i (unscaled)
    double* s_seg;       // [1]
    int* seg_n;          // [max_S]
    unsigned long long* seg_dq;    // [max_S] fixed-point sum of log-ratios, 2^-32 units
    unsigned long long* seg_absq;  // [max_S] coarse sum of |log-ratio|, 2^-8 units
    int* seg_nonfinite;  // [max_S * 3] +inf, -inf, NaN counts
    float* seg_coef;     // [max_S] per-segment gradient coefficient kappa_i
    int* row_counter;    // [1] dynamic row hand-out of the fused kernel; 0 between calls
    long long* cnt_part; // [kRedBlocks] per-block active counts
    double* red_part;    // [kRedBlocks * 4] per-block loss sums
    unsigned* done;      // [3] blocks finished (count, reduce, staged-row); back to 0 after each kernel
    int* err;            // [1]
};

constexpr int kRedBlocks = 64;   // blocks of the count and reduce kernels
static_assert(kRedBlocks % 32 == 0 && kRedBlocks <= 256, "whole warps of block partials, one block of 256 threads");

// Modes of the staged-row kernel: statistics and gradient in one pass; the
// statistics alone (forward only, and the first pass of GSPO); the gradient
// alone from statistics already in the workspace (GSPO's pass after its seam).
enum : int { kModeFused = 0, kModeStats = 1, kModeGrad = 2 };
// row_target of an active row whose target column lies in another vocabulary shard
constexpr int kTargetElsewhere = -2;
constexpr int kMaxShards = 16;

struct CallParams {
    const void* logits;
    const void* teacher;
    void* grad;
    const int64_t* targets;
    const uint8_t* mask;
    int64_t T, V, ld;
    float w_ce, alpha, w_kl;
    // distillation temperature tau: 1 / tau and log2(e) / tau, each rounded once
    // from double (used only by the instantiation for tau != 1)
    float tau_inv, tau_l2;
    int reduction;          // 0 SUM, 1 TOKEN_MEAN
    double inv_denominator; // SUM scale
    const int32_t* seg_ids;
    int num_segments;
    const float* adv;
    const float* old_logp;
    float eps_lo, eps_hi;
    float* loss_out;
    float* logp_out;
    float* lse_out;
    float* kl_out;
    int64_t* count_out;
    int32_t* seg_count_out;
    float* seg_ratio_out;
    uint8_t* seg_flag_out;
    float* seg_loss_out;
    const float* tok_adv;   // GRPO per-token advantages, or null
    float* entropy_out;
    // vocabulary shard: this call's columns are [col0, col0 + V) of v_total
    // (col0 = 0, v_total = V for a whole row)
    int64_t col0, v_total;
    float* part_out;        // shard statistics pass: [T, 4] max, sum, target logit, owns target
    Workspace ws;
    // fused-kernel launch shape and mode
    int mode;               // kModeFused, kModeStats or kModeGrad
    int cluster;
    int64_t slice;          // elements per CTA of a row (multiple of the vector width)
    int nbuf;
    uint32_t buf_bytes;     // bytes of one staged slice
};

__device__ __forceinline__ bool row_active(const CallParams& p, int64_t r, int64_t& t)
{
    t = p.targets[r];
    return t != -100 && (p.mask == nullptr || p.mask[r] != 0);
}

// Target of row r as a column of this call's logits, -100 when the row takes
// no part, kTargetElsewhere when it lies in another vocabulary shard;
// out-of-range targets keep a value outside [0, V) (clamped into int range).
__device__ __forceinline__ int row_target(const CallParams& p, int64_t r)
{
    int64_t t;
    if (!row_active(p, r, t)) return -100;
    if (t < 0) return -1;
    if (t >= p.v_total) return 0x7fffffff;
    t -= p.col0;
    if (t < 0 || t >= p.V) return kTargetElsewhere;
    return static_cast<int>(t);
}

// Cross-entropy scalars of a row from its non-target maximum M, the sum
// S = sum_{j != t} e^(z_j - M) and the target logit, in fp32 with no step
// that cancels:  lse_nt = M + ln S,  d = lse_nt - z_t = (M - z_t) + ln S,
// NLL = softplus(d),  lse = lse_nt + softplus(-d),  and the target's and the
// other columns' probabilities p_t = sigmoid(-d), p_nt = sigmoid(d).
__device__ __forceinline__ void ce_scalars(float M, float S, float zt, float& nll, float& lse, float& lnS,
                                           float& sp_neg, float& pt, float& pnt)
{
    // ln S, e^-|d| and the reciprocal by the fast intrinsics: this chain runs
    // on one lane while the CTA waits for it.  Their errors (ln S a few 1e-7
    // absolute; e^-|d| within 2 + 1.2|d| ulp, under 6e-6 relative while it is a
    // normal number) stay inside the losses' 1e-5.  log1p keeps full precision,
    // since on a confident row the whole NLL is log1p of a tiny e^-|d|.
    lnS = (S == 0.f) ? -INFINITY : __logf(S);
    const float d = (M - zt) + lnS;
    // softplus(+-d) = max(+-d, 0) + log1p(e^-|d|) and sigmoid(+-d) from the
    // same e^-|d|: one exp, one log1p, one division.  The fast exponential
    // flushes results below 2^-126 (|d| above about 87.3) to 0; there the
    // precise one keeps e^-|d| as a subnormal, so a row confident by up to
    // about 103 nats still has a nonzero loss.
    float E = __expf(-fabsf(d));
    if (fabsf(d) > 87.0f) E = expf(-fabsf(d));
    const float l1p = log1pf(E);
    nll = fmaxf(d, 0.f) + l1p;
    sp_neg = fmaxf(-d, 0.f) + l1p;
    lse = (S == 0.f) ? zt : (M + lnS) + sp_neg;
    if (isnan(d)) lse = d;
    const float inv = __fdividef(1.f, 1.f + E);
    pt = (d > 0.f) ? E * inv : inv;
    pnt = (d > 0.f) ? inv : E * inv;
}

// Token scale s: 1/N_active (token mean, 0 if none) or 1/denominator (SUM).
__device__ __forceinline__ float token_scale(const CallParams& p)
{
    if (p.reduction == 1) {
        const int64_t n = *p.ws.n_active;
        return n > 0 ? static_cast<float>(1.0 / static_cast<double>(n)) : 0.f;
    }
    return static_cast<float>(p.inv_denominator);
}

// Interior of columns [c0, c1) of row r that is 16-byte aligned in memory:
// [e0, e1), head [c0, e0), tail [e1, c1).
template <int ESZ>
__device__ __forceinline__ void row_interior(const void* base, int64_t r, int64_t ld, int64_t c0, int64_t c1,
                                             int64_t& e0, int64_t& e1)
{
    const uintptr_t a = reinterpret_cast<uintptr_t>(base) + static_cast<uintptr_t>((r * ld + c0) * ESZ);
    const uintptr_t b = reinterpret_cast<uintptr_t>(base) + static_cast<uintptr_t>((r * ld + c1) * ESZ);
    const uintptr_t a16 = (a + 15) & ~uintptr_t(15);
    const uintptr_t b16 = b & ~uintptr_t(15);
    if (b16 <= a16) { e0 = c1; e1 = c1; return; }
    e0 = c0 + static_cast<int64_t>((a16 - a) / ESZ);
    e1 = c0 + static_cast<int64_t>((b16 - a) / ESZ);
}

// ======================================================================
// K1: fused single-read kernel.
//
// A cluster of C CTAs owns one row at a time; CTA k of the cluster owns the
// columns [k*slice, (k+1)*slice).  Each CTA stages its slice (and the teacher
// slice) in shared memory with one bulk copy per row (nbuf buffers), then
//   pass A: maximum over its non-target columns (packed bf16x2 max), per warp,
//   pass B: sum of 2^((z - m) log2 e) over non-target columns, relative to
//           the warp's maximum (+ teacher max, sum and cross term),
// rebases the warps' partials onto the CTA maximum, pushes one record per CTA
// into every peer's shared memory, and one warp of every CTA merges the
// cluster's records in rank order into the row's fp32 scalars.  Pass C then
// writes the gradient of the slice from the staged copy.  The row is read from
// HBM once and the gradient written once.
//
// Rows are handed out dynamically: rank 0 of each cluster claims the row for
// a later iteration from a global counter and passes it to its peers in its
// record, so clusters that share SMs with others do not set the pace.
// ======================================================================
constexpr int kHdrBytes = 3072;   // mbarriers, row queue, cluster records, warp scratch
constexpr int kMaxCluster = 16;

struct ClusterRec {     // one CTA's partial for the current row (32 bytes; 48 with the entropy
                        // or a teacher)
    float m, s;         // CTA max over its non-target columns; sum e^(z - m)
    float mu, su, w;    // teacher: max, sum e^((u - mu)/tau), sum e^((u - mu)/tau) (u - z) over
                        //   the non-target columns
    float zt;           // target logit (on the CTA that owns the target column)
    int next_row;       // rank 0: row for iteration i + depth (see fused_kernel)
    int next_t;         // rank 0: its target, or -100 when the row is inactive
    float bc;           // sum e^(z - m) (z - m) over the non-target columns (entropy)
    float st;           // tau != 1: sum e^((z - m)/tau) over the non-target columns
    float sunt;         // teacher: su without the target column (w leaves it out too)
    float ut;           // teacher logit at the target (on the owner, 0 elsewhere)
};
static_assert(sizeof(ClusterRec) == 48, "record is two or three 16-byte pushes");

struct RowCoef {        // the row's gradient coefficients, shared by the CTA's threads
    float cz;           // a p_j = sign(a) 2^(z_j log2e - cz)
    float cq;           // teacher: b q_j = 2^(u_j log2e - cq) when b > 0
                        //   (tau != 1: 2^((u_j - mu) Lt - cq), Lt = log2(e) / tau)
    float lseL, luL;    // teacher: p_j = 2^(z_j log2e - lseL), q_j = 2^(u_j log2e - luL)
                        //   (tau != 1: q_j = 2^((u_j - mu) Lt - luL))
    float a, b;         // teacher: g_j = a p_j - b q_j  (tau != 1: a p_j + b (p^tau_j - q_j))
    float gt;           // target column (teacher: minus b q_t still to apply)
    int neg;            // sign of a
    // tau != 1: b p^tau_j = 2^((z_j - mr) Lt - ct), p^tau_j = 2^((z_j - mr) Lt - ltL),
    // with the reference points mr (student) and mu (teacher)
    float ct, ltL, mr, mu;
};

// The row's gradient coefficients (see RowCoef) from its scalars: token scale
// s, lse, the target's CE gradient tg and probability pt, the policy
// coefficient c_r, and with a teacher its Mu and ln Su, and at a temperature the
// tempered student's reference point mr, offset rb and target probability ptt.
// The same arithmetic for the fused pass and for GSPO's gradient pass, which
// reads these scalars back from the workspace.
template <bool KL, bool TAU>
__device__ __forceinline__ RowCoef row_coef(float s, float w_ce, float alpha, float w_kl, float lse, float tg,
                                            float pt, float c_r, float b_kl, float log2_b, bool a_fixed,
                                            float log2_a_fixed, float Mu, float lnSu_g, float mr, float rb,
                                            float ptt)
{
    const float zc = 2.f * alpha * lse;
    const float a = s * (w_ce + zc + (TAU ? 0.f : w_kl)) + c_r;
    RowCoef cf;
    // cz = lse log2e - log2|a|, with the product lse*log2e formed exactly
    const float lseL = lse * kLog2e;
    const float lseL_err = fmaf(lse, kLog2e, -lseL);
    // (a - a) keeps a NaN coefficient (an infinite lse) a NaN
    const float log2_a = a_fixed ? log2_a_fixed + (a - a) : __log2f(fabsf(a));
    cf.cz = (a == 0.f) ? INFINITY : lseL + (lseL_err - log2_a);
    cf.neg = a < 0.f;
    cf.lseL = lseL;
    cf.a = a;
    cf.b = KL ? b_kl : 0.f;
    if (TAU) {
        // b p^tau_j = 2^((z_j - mr) Lt - ct), b q_j = 2^((u_j - Mu) Lt - cq): the
        // exponent offsets stay small, and the products with log2 e exact
        const float rbL = rb * kLog2e, raL = lnSu_g * kLog2e;
        cf.ltL = rbL;
        cf.luL = raL;
        cf.ct = (b_kl > 0.f) ? rbL + (fmaf(rb, kLog2e, -rbL) - log2_b) : INFINITY;
        cf.cq = (b_kl > 0.f) ? raL + (fmaf(lnSu_g, kLog2e, -raL) - log2_b) : INFINITY;
        cf.mr = mr;
        cf.mu = Mu;
        cf.gt = (s * w_ce + c_r) * tg + s * zc * pt + b_kl * ptt;
    } else if (KL) {
        const float lu = Mu + lnSu_g;   // teacher's logsumexp
        const float luL = lu * kLog2e;
        cf.luL = luL;
        cf.cq = (b_kl > 0.f) ? luL + (fmaf(lu, kLog2e, -luL) - log2_b) : INFINITY;
        cf.ct = INFINITY;
        cf.ltL = 0.f;
        cf.mr = 0.f;
        cf.mu = 0.f;
        cf.gt = (s * w_ce + c_r) * tg + s * (zc + w_kl) * pt;
    } else {
        cf.luL = 0.f;
        cf.cq = INFINITY;
        cf.ct = INFINITY;
        cf.ltL = 0.f;
        cf.mr = 0.f;
        cf.mu = 0.f;
        cf.gt = (s * w_ce + c_r) * tg + s * zc * pt;
    }
    return cf;
}

// The same for GSPO's gradient pass, out of line: that pass runs in the same
// instantiation as the fused one, whose merge this keeps as it was.
template <bool KL, bool TAU>
__device__ __noinline__ RowCoef row_coef_grad(float s, float w_ce, float alpha, float w_kl, float lse, float tg,
                                              float pt, float c_r, float b_kl, float log2_b, float Mu,
                                              float lnSu_g, float mr, float rb, float ptt)
{
    return row_coef<KL, TAU>(s, w_ce, alpha, w_kl, lse, tg, pt, c_r, b_kl, log2_b, false, 0.f, Mu, lnSu_g, mr, rb,
                             ptt);
}

template <class IO, int NT>
__device__ __noinline__ float sum_ea_guarded(uint32_t bz, int nvec, int tid, int vt, int kt, float mL);

// Pass B sums over the staged interior, target column excluded, with
// e = 2^a and a = z log2e - mL (mL the slice maximum in base 2):
//   s = sum e,   b = sum e a  (only with ENT: the entropy partial).
// A logit of -inf gives e = 0 and e a = NaN in the packed loop; a thread that
// met one redoes its columns with the guard, which costs nothing otherwise.
template <class IO, int NT, bool ENT>
__device__ __forceinline__ void sums_plain(uint32_t bz, int nvec, int tid, int vt, int kt, float mL,
                                           float& s_out, float& b_out)
{
    constexpr int VN = IO::N;
    const uint64_t L2 = f2_pack(kLog2e, kLog2e);
    const uint64_t nm2 = f2_pack(-mL, -mL);
    uint64_t acc = f2_pack(0.f, 0.f), accb = acc;
    float s0 = 0.f, b0 = 0.f;
#pragma unroll 2
    for (int v = tid; v < nvec; v += NT) {
        const uint4 q = lds128(bz + v * 16);
        if (v != vt) {
            // packed pairs: one f32x2 FMA forms two exponent arguments, one
            // f32x2 add accumulates two terms
#pragma unroll
            for (int k = 0; k < VN / 2; ++k) {
                const uint64_t arg = f2_fma(IO::pair(q, k), L2, nm2);
                float a0, a1;
                f2_unpack(arg, a0, a1);
                const uint64_t e = f2_pack(ex2(a0), ex2(a1));
                acc = f2_add(acc, e);
                if (ENT) accb = f2_fma(e, arg, accb);
            }
        } else {
            float x[VN];
            IO::unpack(q, x);
#pragma unroll
            for (int j = 0; j < VN; ++j)
                if (j != kt) {
                    const float a = fmaf(x[j], kLog2e, -mL);
                    const float e = ex2(a);
                    s0 += e;
                    if (ENT && e > 0.f) b0 = fmaf(e, a, b0);
                }
        }
    }
    float h0, h1;
    f2_unpack(acc, h0, h1);
    s_out = s0 + (h0 + h1);
    if (ENT) {
        f2_unpack(accb, h0, h1);
        b0 += h0 + h1;
        if (isnan(b0) && !isnan(s_out)) b0 = sum_ea_guarded<IO, NT>(bz, nvec, tid, vt, kt, mL);
    }
    b_out = b0;
}

// The same with the teacher slice (guard-free form: a -inf teacher logit makes
// w NaN, and the caller then takes w again with sum_w_guarded), the target
// column left out like the student's:
//   su = sum 2^c, c = u Lt - muL,   w = sum 2^c (u - z),   et = 2^c of the target,
// with Lt = log2e, or log2(e) / tau at a temperature (TAU), where the student's
// non-target sum at the temperature is taken too:  st = sum 2^(z Lt - mLt).
template <class IO, int NT, bool ENT, bool TAU>
__device__ __forceinline__ void sums_kl(uint32_t bz, uint32_t bu, int nvec, int tid, int vt, int kt, float mL,
                                        float muL, float Lt, float mLt, float& s_out, float& su_out,
                                        float& w_out, float& b_out, float& st_out, float& et_out)
{
    constexpr int VN = IO::N;
    const uint64_t L2 = f2_pack(kLog2e, kLog2e);
    const uint64_t Lt2 = TAU ? f2_pack(Lt, Lt) : L2;
    const uint64_t nm2 = f2_pack(-mL, -mL);
    const uint64_t nmu2 = f2_pack(-muL, -muL);
    const uint64_t nmt2 = f2_pack(-mLt, -mLt);
    const uint64_t neg1 = f2_pack(-1.f, -1.f);
    uint64_t accz = f2_pack(0.f, 0.f), accu = accz, accw = accz, accb = accz, acct = accz;
    float et = 0.f;
    // one vector: the student terms of every column but lane `kill` (the
    // target's, or -1), the teacher terms of every column
    auto vec = [&](int v, int kill) {
        const uint4 q = lds128(bz + v * 16);
        const uint4 qu = lds128(bu + v * 16);
#pragma unroll
        for (int k = 0; k < VN / 2; ++k) {
            const uint64_t xz = IO::pair(q, k), xu = IO::pair(qu, k);
            float a0, a1, u0, u1;
            const uint64_t argz = f2_fma(xz, L2, nm2);
            f2_unpack(argz, a0, a1);
            f2_unpack(f2_fma(xu, Lt2, nmu2), u0, u1);
            float e0 = ex2(a0), e1 = ex2(a1);
            if (2 * k == kill) e0 = 0.f;
            if (2 * k + 1 == kill) e1 = 0.f;
            const uint64_t ez = f2_pack(e0, e1);
            accz = f2_add(accz, ez);
            if (ENT) accb = f2_fma(ez, argz, accb);
            if (TAU) {
                float t0, t1;
                f2_unpack(f2_fma(xz, Lt2, nmt2), t0, t1);
                float f0 = ex2(t0), f1 = ex2(t1);
                if (2 * k == kill) f0 = 0.f;
                if (2 * k + 1 == kill) f1 = 0.f;
                acct = f2_add(acct, f2_pack(f0, f1));
            }
            float g0 = ex2(u0), g1 = ex2(u1);
            if (2 * k == kill) { et = g0; g0 = 0.f; }
            if (2 * k + 1 == kill) { et = g1; g1 = 0.f; }
            const uint64_t eu = f2_pack(g0, g1);
            accu = f2_add(accu, eu);
            accw = f2_fma(eu, f2_fma(xz, neg1, xu), accw);   // e^((u-mu)/tau) (u - z)
        }
    };
    // the target's vector is taken out of the loop, so the loop body needs no
    // per-column test
#pragma unroll 2
    for (int v = tid; v < nvec; v += NT)
        if (v != vt) vec(v, -1);
    if (vt >= 0 && vt % NT == tid) vec(vt, kt);
    float h0, h1;
    f2_unpack(accz, h0, h1);
    s_out = h0 + h1;
    f2_unpack(accu, h0, h1);
    su_out = h0 + h1;
    f2_unpack(accw, h0, h1);
    w_out = h0 + h1;
    f2_unpack(acct, h0, h1);
    st_out = TAU ? h0 + h1 : 0.f;
    et_out = et;
    float b0 = 0.f;
    if (ENT) {
        f2_unpack(accb, h0, h1);
        b0 = h0 + h1;
        if (isnan(b0) && !isnan(s_out)) b0 = sum_ea_guarded<IO, NT>(bz, nvec, tid, vt, kt, mL);
    }
    b_out = b0;
}

// b = sum e a over this thread's columns of the interior, skipping e = 0.
template <class IO, int NT>
__device__ __noinline__ float sum_ea_guarded(uint32_t bz, int nvec, int tid, int vt, int kt, float mL)
{
    constexpr int VN = IO::N;
    float b = 0.f;
    for (int v = tid; v < nvec; v += NT) {
        float x[VN];
        IO::unpack(lds128(bz + v * 16), x);
        for (int j = 0; j < VN; ++j) {
            const float a = fmaf(x[j], kLog2e, -mL);
            const float e = ex2(a);
            if ((v != vt || j != kt) && e > 0.f) b = fmaf(e, a, b);
        }
    }
    return b;
}

// w = sum 2^c (u - z), c = u Lt - muL, over this thread's non-target columns
// of the interior, skipping 2^c = 0.
template <class IO, int NT>
__device__ __noinline__ float sum_w_guarded(uint32_t bz, uint32_t bu, int nvec, int tid, int vt, int kt, float muL,
                                            float Lt)
{
    constexpr int VN = IO::N;
    float w = 0.f;
    for (int v = tid; v < nvec; v += NT) {
        float x[VN], y[VN];
        IO::unpack(lds128(bz + v * 16), x);
        IO::unpack(lds128(bu + v * 16), y);
        for (int j = 0; j < VN; ++j) {
            const float eu = ex2(fmaf(y[j], Lt, -muL));
            if (eu > 0.f && (v != vt || j != kt)) w = fmaf(eu, y[j] - x[j], w);
        }
    }
    return w;
}

// Occupancy: without a teacher, shared memory admits 1024 threads per SM at the
// default shape; with one, two CTAs share an SM, so registers are capped to fit two.
template <bool KL, int NT>
constexpr int fused_min_blocks() { return NT >= 1024 ? 1 : (KL ? 2 : 1024 / NT); }

// EARLY: the statistics pass (no gradient), which hands its buffer to the next
// copy as soon as pass B is done; a separate instantiation, so that the passes
// that write the gradient compile exactly as without it.
// TAU: distillation at a temperature tau != 1 (with KL only).  The teacher's
// exponentials take the factor log2(e) / tau, and the student's tempered
// distribution p^tau = softmax(z / tau) is a third sum next to the cross-entropy's
// and the teacher's, so that its gradient term w_kl (p^tau - q) / tau is a
// third exponential in pass C.  A separate instantiation, so that tau = 1
// compiles exactly as without it.
// ENT (without a teacher only): the per-row entropy output is requested
// (entropy_out != null); without it no entropy partial is summed, reduced or
// exchanged.  With a teacher the entropy is decided at run time and the
// partial's butterflies run on zeros when it is not wanted: measured, the
// compile-time form made that instantiation 1.5-1.8% slower, where it made the
// plain one 1.8% faster.
template <bool BF16, bool KL, int NT, bool EARLY, bool TAU, bool ENT>
__global__ void __launch_bounds__(NT, (fused_min_blocks<KL, NT>())) fused_kernel(const CallParams p)
{
    static_assert(KL || !TAU, "a temperature needs a teacher");
    static_assert(!(KL && ENT), "with a teacher the entropy is decided at run time");
    // the entropy wanted: read from the parameters at each use (not held in a
    // register through the row loop)
#define LMLOSS_ENT_RT (KL ? (p.entropy_out != nullptr) : ENT)
    using IO = Vec<BF16>;
    constexpr int VN = IO::N;
    constexpr int ESZ = IO::ESZ;
    constexpr int NW = NT / 32;
    static_assert(NW <= 32, "at most 32 warps");
    // butterflies over the warps' partials (lanes 0..NW-1) and over the cluster's
    // records (lanes 0..C-1, C <= 16): lanes 0..15 already hold the full result
    // after the rounds below 16 when at most 16 lanes carry values, and lanes
    // 0..C-1 are the ones that use it
    constexpr int kPubOff = NW > 16 ? 16 : 8;
    constexpr int kRecOff = kMaxCluster / 2;
    static_assert(kMaxCluster == 16, "record butterflies cover lanes 0..15");

    extern __shared__ __align__(128) unsigned char smem[];
    uint64_t* mbar = reinterpret_cast<uint64_t*>(smem);                  // [2] staged-row copies
    uint64_t* rbar = reinterpret_cast<uint64_t*>(smem + 16);             // [2] cluster records, by row parity
    int* rowq = reinterpret_cast<int*>(smem + 32);                       // [4] row of iteration i (i & 3)
    int* tq = reinterpret_cast<int*>(smem + 48);                         // [4] its target (-100: inactive)
    float* slot = reinterpret_cast<float*>(smem + 64);                   // [1] target logit
    RowCoef* coef = reinterpret_cast<RowCoef*>(smem + 96);               // [1]
    float* wred = reinterpret_cast<float*>(smem + 256);                  // [8][32]
    ClusterRec* rec = reinterpret_cast<ClusterRec*>(smem + 1280);        // [2][kMaxCluster]
    unsigned char* bufs = smem + kHdrBytes;

    const int tid = threadIdx.x;
    const int lane = tid & 31, warp = tid >> 5;
    const uint32_t rank = cluster_rank();
    const int C = p.cluster;
    const int cid = static_cast<int>(blockIdx.x) / C;
    const int G = static_cast<int>(gridDim.x) / C;
    const int64_t c0 = min(p.V, static_cast<int64_t>(rank) * p.slice);
    const int64_t c1 = min(p.V, c0 + p.slice);
    const int nbuf = p.nbuf;
    // Rows known ahead of the one in hand.  A pass that writes the gradient
    // frees a buffer at the end of the row (the copy of row i + nbuf - 1 goes
    // out at the top of row i); the statistics pass frees it after pass B, so
    // the copy of row i + nbuf goes out then, under the record exchange, and
    // the row after it must already be known.
    constexpr bool early = EARLY;   // launched only with mode == kModeStats
    const int depth = nbuf + (early ? 1 : 0);
    const float s_tok = token_scale(p);
    // Kernel-wide constants of the row coefficients: b = s w_kl / tau and, when
    // no per-row term enters it (no z-loss, no policy term), a = s (w_ce + w_kl)
    // at tau = 1 (where p^tau = p), a = s w_ce otherwise.
    const float b_kl = s_tok * p.w_kl * (TAU ? p.tau_inv : 1.f);
    const float log2_b = (b_kl > 0.f) ? log2f(b_kl) : 0.f;
    const bool a_fixed = p.alpha == 0.f && !p.tok_adv;   // (GSPO's gradient pass does not use it)
    const float log2_a_fixed = log2f(fabsf(s_tok * (p.w_ce + (TAU ? 0.f : p.w_kl))));
    // base-2 factor of the teacher's exponentials (and of the student's at the temperature)
    const float Lt = TAU ? p.tau_l2 : kLog2e;
    const int mode = p.mode;

    auto buf_addr = [&](int b, int a) -> uint32_t {
        return smem_addr(bufs + (static_cast<size_t>(b) * (KL ? 2 : 1) + a) * p.buf_bytes);
    };
    auto bar_addr = [&](int b) -> uint32_t { return smem_addr(&mbar[b]); };

    if (tid == 0) {
        for (int b = 0; b < nbuf; ++b) mbar_init(bar_addr(b), 1);
        mbar_init(smem_addr(&rbar[0]), 1);
        mbar_init(smem_addr(&rbar[1]), 1);
        for (int k = 0; k < 4; ++k) {
            rowq[k] = (k < depth) ? cid + k * G : 0x7fffffff;
            tq[k] = (k < depth && rowq[k] < p.T) ? row_target(p, rowq[k]) : -100;
        }
        fence_mbar_init();
    }
    cluster_sync_all();   // every peer's record barriers exist before anyone pushes

    // Producer side (thread 0): stage row rr's slice into buffer b.
    auto issue = [&](int64_t rr, int tt, int b) {
        const bool act = tt != -100;
        int64_t e0, e1;
        row_interior<ESZ>(p.logits, rr, p.ld, c0, c1, e0, e1);
        const uint32_t bytes = static_cast<uint32_t>((e1 - e0) * ESZ);
        if (!act || bytes == 0) {
            mbar_arrive(bar_addr(b));
            return;
        }
        mbar_arrive_expect_tx(bar_addr(b), bytes * (KL ? 2u : 1u));
        const size_t off = static_cast<size_t>(rr * p.ld + e0) * ESZ;
        bulk_load(buf_addr(b, 0), static_cast<const unsigned char*>(p.logits) + off, bytes, bar_addr(b));
        if (KL)
            bulk_load(buf_addr(b, 1), static_cast<const unsigned char*>(p.teacher) + off, bytes, bar_addr(b));
    };

    if (tid == 0)
        for (int k = 0; k < (early ? nbuf : nbuf - 1); ++k)
            if (rowq[k] < p.T) issue(rowq[k], tq[k], k);

    bool failed = false;
    for (int i = 0;; ++i) {
        const int64_t r = rowq[i & 3];
        if (r >= p.T) break;
        __syncthreads();   // buffers, scratch and coefficients of the previous row are free
        int claim_row = 0;
        if (tid == 0) {
            const int j = (i + nbuf - 1) & 3;
            if (!early && rowq[j] < p.T) issue(rowq[j], tq[j], (i + nbuf - 1) % nbuf);
            if (rank == 0) claim_row = depth * G + atomicAdd(p.ws.row_counter, 1);
        }
        const int b = i % nbuf;
        const uint32_t parity = static_cast<uint32_t>((i / nbuf) & 1);

        const int64_t t = tq[i & 3];
        const bool act = t != -100;
        const bool elsewhere = t == kTargetElsewhere;   // target in another vocabulary shard
        const bool bad = act && !elsewhere && (t < 0 || t >= p.V);
        int64_t e0, e1;
        row_interior<ESZ>(p.logits, r, p.ld, c0, c1, e0, e1);
        const int nvec = static_cast<int>((e1 - e0) / VN);
        const size_t row_off = static_cast<size_t>(r * p.ld) * ESZ;
        const uint32_t bz = buf_addr(b, 0);
        const uint32_t bu = KL ? buf_addr(b, 1) : 0u;
        const int64_t tv = t - e0;   // target offset within the interior (may be outside)
        const bool owner = act && t >= c0 && t < c1;
        // the one interior vector holding the target (-1 if none) and its lane
        const int vt = (act && tv >= 0 && tv < static_cast<int64_t>(nvec) * VN) ? static_cast<int>(tv / VN) : -1;
        const int kt = (vt >= 0) ? static_cast<int>(tv - static_cast<int64_t>(vt) * VN) : -1;

        if (!failed && !mbar_wait_bounded(bar_addr(b), parity, kWaitLimitCycles)) {
            set_error(p.ws.err, kErrTimeout);
            failed = true;
        }

        // the claimed row's target: loaded now, while the passes run, because the
        // whole cluster waits on rank 0's record that carries it
        int next_t_pf = -100;
        if (tid == 0 && rank == 0 && claim_row < p.T) next_t_pf = row_target(p, claim_row);

        // Per-row inputs of the merge: GRPO's advantage and old log-prob, and in
        // GSPO's gradient pass the row's statistics and segment coefficient from
        // the workspace.  With a teacher they are loaded here, their latency under
        // the passes;
        // without one, where the merge uses them (measured on GB300: the early
        // loads cost the teacher-free kernel 1.8% even when neither term is in
        // the call, and saved the teacher kernel as much)
        float g_lse = 0.f, g_nll = 0.f, g_cr = 0.f, g_adv = 0.f, g_old = 0.f;
        auto load_policy = [&]() {
            g_adv = p.tok_adv[r];
            g_old = p.old_logp[r];
        };
        auto load_grad = [&]() {
            g_lse = p.ws.row_lse[r];
            g_nll = p.ws.row_nll[r];
            const int gs = p.seg_ids ? p.seg_ids[r] : -1;
            g_cr = (gs >= 0 && gs < p.num_segments) ? p.ws.seg_coef[gs] : 0.f;
        };
        if (KL && p.tok_adv && mode != kModeGrad && warp == 0 && lane == 0 && act && !bad) load_policy();
        if (KL && mode == kModeGrad && warp == 0 && lane == 0 && act && !bad) load_grad();

        // ---- pass A: maxima (non-target for z, all columns for u), per warp: each
        // warp takes its sums against its own maxima and the warps' partials are
        // rebased once, when the CTA's record is built, so no CTA barrier sits
        // between the two passes
        // (the thread holding the target column also records the target's logit,
        // and with a teacher the teacher's, for the merge)
        float m_w = -INFINITY, mu_w = -INFINITY;
        if (act && mode != kModeGrad) {
            uint32_t accz = IO::max_init(), accu = IO::max_init();
            float mx = -INFINITY, mu = -INFINITY;
#pragma unroll 4
            for (int v = tid; v < nvec; v += NT) {
                const uint4 q = lds128(bz + v * 16);
                if (v == vt) {
                    float x[VN];
                    IO::unpack(q, x);
#pragma unroll
                    for (int j = 0; j < VN; ++j) {
                        if (j != kt) mx = fmaxf(mx, x[j]);
                        else slot[0] = x[j];
                    }
                    if (KL) {
                        float y[VN];
                        IO::unpack(lds128(bu + v * 16), y);
#pragma unroll
                        for (int j = 0; j < VN; ++j)
                            if (j == kt) slot[1] = y[j];
                    }
                } else {
                    accz = IO::max_acc(accz, q);
                }
                if (KL) {
                    const uint4 qu = lds128(bu + v * 16);
                    accu = IO::max_acc(accu, qu);
                }
            }
            if (tid == NT - 1) {
                for (int pass = 0; pass < 2; ++pass) {
                    const int64_t lo = pass == 0 ? c0 : e1, hi = pass == 0 ? e0 : c1;
                    for (int64_t j = lo; j < hi; ++j) {
                        const float x = IO::load1(p.logits, r * p.ld + j);
                        if (j != t) mx = fmaxf(mx, x);
                        else slot[0] = x;
                        if (KL) {
                            const float y = IO::load1(p.teacher, r * p.ld + j);
                            mu = fmaxf(mu, y);
                            if (j == t) slot[1] = y;
                        }
                    }
                }
            }
            float m = fmaxf(IO::max_final(accz), mx);
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
            if (KL) {
                mu = fmaxf(mu, IO::max_final(accu));
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) mu = fmaxf(mu, __shfl_xor_sync(0xffffffffu, mu, off));
            }
            m_w = m;
            if (KL) mu_w = mu;
        }

        // ---- pass B: sums relative to the warp's maxima
        if (act && mode != kModeGrad) {
            const float mL = (m_w == -INFINITY) ? 0.f : m_w * kLog2e;
            const float muL = (mu_w == -INFINITY) ? 0.f : mu_w * Lt;
            const float mLt = (!TAU || m_w == -INFINITY) ? 0.f : m_w * Lt;
            float s0 = 0.f, s1 = 0.f, su = 0.f, w = 0.f, b0 = 0.f, st = 0.f, et = 0.f;
            if (!KL) sums_plain<IO, NT, ENT>(bz, nvec, tid, vt, kt, mL, s0, b0);
            if (KL) {
                if (LMLOSS_ENT_RT)
                    sums_kl<IO, NT, true, TAU>(bz, bu, nvec, tid, vt, kt, mL, muL, Lt, mLt, s0, su, w, b0, st, et);
                else
                    sums_kl<IO, NT, false, TAU>(bz, bu, nvec, tid, vt, kt, mL, muL, Lt, mLt, s0, su, w, b0, st, et);
                // a -inf teacher logit gives 0 * -inf = NaN in the guard-free cross
                // term: a thread that met one takes that sum again with the guard
                if (isnan(w) && !isnan(su)) w = sum_w_guarded<IO, NT>(bz, bu, nvec, tid, vt, kt, muL, Lt);
            }
            float s = s0 + s1;
            if (tid == NT - 1) {
                for (int pass = 0; pass < 2; ++pass) {
                    const int64_t lo = pass == 0 ? c0 : e1, hi = pass == 0 ? e0 : c1;
                    for (int64_t j = lo; j < hi; ++j) {
                        const float x = IO::load1(p.logits, r * p.ld + j);
                        if (j != t) {
                            const float a = fmaf(x, kLog2e, -mL);
                            const float e = ex2(a);
                            s += e;
                            if (e > 0.f) b0 = fmaf(e, a, b0);
                            if (TAU) st += ex2(fmaf(x, Lt, -mLt));
                        }
                        if (KL) {
                            const float y = IO::load1(p.teacher, r * p.ld + j);
                            const float eu = ex2(fmaf(y, Lt, -muL));
                            if (j != t) {
                                su += eu;
                                w += (eu > 0.f) ? eu * (y - x) : 0.f;
                            } else {
                                et = eu;
                            }
                        }
                    }
                }
            }
            // the teacher's sum over all columns (sua: the target's term folded back
            // in, for the gradient) and without the target (su, for the KL)
            float sua = su + et;
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) {
                s += __shfl_xor_sync(0xffffffffu, s, off);
                if (ENT || KL) b0 += __shfl_xor_sync(0xffffffffu, b0, off);   // see ENT
                if (KL) {
                    su += __shfl_xor_sync(0xffffffffu, su, off);
                    sua += __shfl_xor_sync(0xffffffffu, sua, off);
                    w += __shfl_xor_sync(0xffffffffu, w, off);
                }
                if (TAU) st += __shfl_xor_sync(0xffffffffu, st, off);
            }
            if (lane == 0) {
                wred[warp] = m_w;
                wred[64 + warp] = s;
                wred[192 + warp] = b0;
                if (KL) { wred[32 + warp] = mu_w; wred[96 + warp] = sua; wred[128 + warp] = w; wred[224 + warp] = su; }
                if (TAU) wred[160 + warp] = st;
            }
        }
        __syncthreads();

        // statistics pass: every thread is done with this buffer (passes A and B,
        // after its wait), so it takes the copy of row i + nbuf now; the last
        // warp issues it, leaving warp 0 free to publish the record
        if (early && tid == NT - 32) {
            const int j = (i + nbuf) & 3;
            if (rowq[j] < p.T) issue(rowq[j], tq[j], b);
        }

        // ---- publish this CTA's record
        if (warp == 0) {
            float s = 0.f, su = 0.f, sun = 0.f, w = 0.f, bc = 0.f, st = 0.f;
            float m_cta = -INFINITY, mu_cta = -INFINITY;
            if (act) {
                // warp w's sums are against round(m_w log2e): rebase them onto
                // round(m_cta log2e) (entropy partial: e (a + d) summed = f (b + s d))
                const float mw = (lane < NW) ? wred[lane] : -INFINITY;
                m_cta = mw;
#pragma unroll
                for (int off = kPubOff; off > 0; off >>= 1) m_cta = fmaxf(m_cta, __shfl_xor_sync(0xffffffffu, m_cta, off));
                const float mLc = (m_cta == -INFINITY) ? 0.f : m_cta * kLog2e;
                const float mLw = (mw == -INFINITY) ? 0.f : mw * kLog2e;
                s = (lane < NW) ? wred[64 + lane] : 0.f;
                const float dz = mLw - mLc;
                const float fz = (s == 0.f) ? 0.f : ex2(dz);
                if (ENT || KL) {
                    bc = (lane < NW) ? wred[192 + lane] : 0.f;
                    bc = (s == 0.f) ? 0.f : fz * fmaf(s, dz, bc);
                }
                s *= fz;
                if (TAU) {
                    // the tempered sum likewise, against round(m Lt)
                    st = (lane < NW) ? wred[160 + lane] : 0.f;
                    const float mLtc = (m_cta == -INFINITY) ? 0.f : m_cta * Lt;
                    const float mLtw = (mw == -INFINITY) ? 0.f : mw * Lt;
                    st = (st == 0.f) ? 0.f : st * ex2(mLtw - mLtc);
                }
                if (KL) {
                    const float muw = (lane < NW) ? wred[32 + lane] : -INFINITY;
                    mu_cta = muw;
#pragma unroll
                    for (int off = kPubOff; off > 0; off >>= 1)
                        mu_cta = fmaxf(mu_cta, __shfl_xor_sync(0xffffffffu, mu_cta, off));
                    const float muLc = (mu_cta == -INFINITY) ? 0.f : mu_cta * Lt;
                    const float muLw = (muw == -INFINITY) ? 0.f : muw * Lt;
                    su = (lane < NW) ? wred[96 + lane] : 0.f;
                    sun = (lane < NW) ? wred[224 + lane] : 0.f;
                    w = (lane < NW) ? wred[128 + lane] : 0.f;
                    const float fu = (su == 0.f) ? 0.f : ex2(muLw - muLc);
                    su *= fu;
                    sun *= fu;
                    w *= fu;
                }
#pragma unroll
                for (int off = kPubOff; off > 0; off >>= 1) {
                    s += __shfl_xor_sync(0xffffffffu, s, off);
                    if (ENT || KL) bc += __shfl_xor_sync(0xffffffffu, bc, off);
                    if (KL) {
                        su += __shfl_xor_sync(0xffffffffu, su, off);
                        sun += __shfl_xor_sync(0xffffffffu, sun, off);
                        w += __shfl_xor_sync(0xffffffffu, w, off);
                    }
                    if (TAU) st += __shfl_xor_sync(0xffffffffu, st, off);
                }
            }
            // lanes 0..15 hold the CTA totals and build the same record; lane c
            // pushes it into slot [i & 1][rank] of CTA c, whose record barrier for
            // this parity counts the bytes
            const int claim_b = __shfl_sync(0xffffffffu, claim_row, 0);
            const int next_t_b = __shfl_sync(0xffffffffu, next_t_pf, 0);
            ClusterRec R;
            // the sums were taken against round(m log2e); undo that rounding exactly
            const float mL = (m_cta == -INFINITY) ? 0.f : m_cta * kLog2e;
            const float muL = (mu_cta == -INFINITY) ? 0.f : mu_cta * Lt;
            R.m = m_cta;
            // e = 2^(z log2e - mL) = e^(z - m) 2^delta and bc sums e (z log2e - mL), so
            // sum e^(z - m) (z - m) = 2^-delta (bc - delta s) / log2e
            const float delta = (m_cta == -INFINITY) ? 0.f : fmaf(m_cta, kLog2e, -mL);
            const float f = ex2(-delta);
            R.s = s * f;
            R.bc = (bc - delta * s) * f * (1.0f / kLog2e);
            R.st = 0.f;
            if (TAU) {
                const float mLt = (m_cta == -INFINITY) ? 0.f : m_cta * Lt;
                R.st = st * ((m_cta == -INFINITY) ? 1.f : ex2(-fmaf(m_cta, Lt, -mLt)));
            }
            R.mu = mu_cta;
            const float fu = (mu_cta == -INFINITY) ? 1.f : ex2(-fmaf(mu_cta, Lt, -muL));
            R.su = su * fu;
            R.sunt = sun * fu;
            R.w = w * fu;
            R.zt = owner ? slot[0] : 0.f;   // exactly 0 in every CTA but the target's owner
            R.ut = (KL && owner) ? slot[1] : 0.f;
            R.next_row = (rank == 0) ? claim_b : 0;
            R.next_t = (rank == 0) ? next_t_b : -100;
            const uint4* Rv = reinterpret_cast<const uint4*>(&R);
            const uint32_t my_slot = smem_addr(&rec[(i & 1) * kMaxCluster + rank]);
            const uint32_t my_bar = smem_addr(&rbar[i & 1]);
            // the third 16 bytes (entropy partial; with a teacher the target's
            // terms and the tempered sum) travel only when used
            constexpr bool ent = KL || ENT;
            const uint32_t rec_bytes = ent ? 48u : 32u;
            if (lane == 0) mbar_arrive_expect_tx(my_bar, static_cast<uint32_t>(C) * rec_bytes);
            if (lane < C) {
                const uint32_t dst = dsmem_map(my_slot, static_cast<uint32_t>(lane));
                const uint32_t bar = dsmem_map(my_bar, static_cast<uint32_t>(lane));
                st_async_v4(dst, Rv[0], bar);
                st_async_v4(dst + 16, Rv[1], bar);
                if (ent) st_async_v4(dst + 32, Rv[2], bar);
            }
        }

        // ---- merge the cluster's records (one warp), row scalars in fp32
        if (warp == 0) {
            if (!failed && !mbar_wait_cluster_bounded(smem_addr(&rbar[i & 1]), static_cast<uint32_t>((i >> 1) & 1),
                                                      kWaitLimitCycles)) {
                set_error(p.ws.err, kErrTimeout);
                failed = true;
            }
            ClusterRec q;
            q.m = -INFINITY; q.s = 0.f; q.mu = -INFINITY; q.su = 0.f; q.w = 0.f; q.zt = 0.f;
            q.next_row = 0; q.next_t = -100; q.bc = 0.f; q.st = 0.f; q.sunt = 0.f; q.ut = 0.f;
            if (lane < C) q = rec[(i & 1) * kMaxCluster + lane];
            const int next_row = __shfl_sync(0xffffffffu, q.next_row, 0);
            const int next_t = __shfl_sync(0xffffffffu, q.next_t, 0);
            if (bad && rank == 0 && lane == 0 && mode != kModeGrad) set_error(p.ws.err, kErrBadTarget);
            // (the statistics instantiation never runs GSPO's gradient mode, and only
            // it runs the vocabulary shards' statistics pass: each branch is compiled
            // where it can be taken)
            if (!EARLY && act && mode == kModeGrad) {
                if (lane == 0) {
                    if (!KL && !bad) load_grad();
                    // s (w_ce (p - onehot) + 2 alpha lse p) + c_r (p - onehot)
                    const float nll = bad ? __int_as_float(0x7fc00000) : g_nll;
                    const float lse = bad ? nll : g_lse;
                    const float pt = expf(-nll);
                    const float tg = (pt < 0.25f) ? pt - 1.0f : expm1f(-nll);
                    // with a teacher, its statistics from the statistics pass (loaded here,
                    // not with the others above: the fused pass shares this code and
                    // keeps its registers for the row's sweeps)
                    float2 g_tu = make_float2(0.f, 0.f);
                    float4 g_tt = make_float4(0.f, 0.f, 0.f, 0.f);
                    if (KL && !bad) g_tu = reinterpret_cast<const float2*>(p.ws.row_tu)[r];
                    if (TAU && !bad) g_tt = reinterpret_cast<const float4*>(p.ws.row_tt)[r];
                    *coef = row_coef_grad<KL, TAU>(s_tok, p.w_ce, p.alpha, p.w_kl, lse, tg, pt, g_cr, b_kl, log2_b,
                                                   g_tu.x, g_tu.y, g_tt.x, g_tt.y, g_tt.z);
                }
            } else if (act) {
                float M = q.m;
#pragma unroll
                for (int off = kRecOff; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
                const float fz = rescale(q.m, M);
                float S = q.s * fz;
                // sum e^(z - M) (z - M) over this CTA's non-target columns
                float Bc = (!LMLOSS_ENT_RT || q.s == 0.f) ? 0.f : fz * (q.bc + q.s * (q.m - M));
                float Zt = q.zt;   // summed below: every record but the owner's holds exactly 0
                float Mu = q.mu, Su = 0.f, Sun = 0.f, W = 0.f;
                float Ut = q.ut;   // summed like Zt
                float St = TAU ? q.st * rescale(q.m, M, Lt) : 0.f;
                if (KL) {
#pragma unroll
                    for (int off = kRecOff; off > 0; off >>= 1) Mu = fmaxf(Mu, __shfl_xor_sync(0xffffffffu, Mu, off));
                    const float f = rescale(q.mu, Mu, Lt);
                    Su = q.su * f;
                    Sun = q.sunt * f;
                    W = q.w * f;
                }
#pragma unroll
                for (int off = kRecOff; off > 0; off >>= 1) {
                    S += __shfl_xor_sync(0xffffffffu, S, off);
                    if (LMLOSS_ENT_RT) Bc += __shfl_xor_sync(0xffffffffu, Bc, off);
                    Zt += __shfl_xor_sync(0xffffffffu, Zt, off);
                    if (KL) {
                        Su += __shfl_xor_sync(0xffffffffu, Su, off);
                        Sun += __shfl_xor_sync(0xffffffffu, Sun, off);
                        W += __shfl_xor_sync(0xffffffffu, W, off);
                        Ut += __shfl_xor_sync(0xffffffffu, Ut, off);
                    }
                    if (TAU) St += __shfl_xor_sync(0xffffffffu, St, off);
                }
                const float ztf = Zt;
                if (EARLY && p.part_out) {
                    // vocabulary shard, statistics pass: the shard's partials go out as they
                    // are and are merged across shards by shard_merge_kernel
                    if (lane == 0 && rank == 0) {
                        float* o = p.part_out + 4 * r;
                        o[0] = M;
                        o[1] = S;
                        o[2] = ztf;
                        o[3] = (!bad && !elsewhere) ? 1.f : 0.f;
                    }
                } else if (lane == 0) {
                    // fp32 throughout, arranged so that no step cancels:
                    //   lse_nt = M + ln S,  d = lse_nt - z_t = (M - z_t) + ln S  (M - z_t exact),
                    //   NLL = softplus(d),  lse = lse_nt + softplus(-d)
                    const float zt = bad ? __int_as_float(0x7fc00000) : ztf;
                    float nll, lse, lnS, sp_neg, pt, pnt;
                    ce_scalars(M, S, zt, nll, lse, lnS, sp_neg, pt, pnt);
                    const float tg = (pt < 0.25f) ? pt - 1.0f : -pnt;
                    // KL = sum q (log q - log p^tau) with log q_j = (u_j - Mu)/tau - ln Su
                    // and log p^tau_j = (z_j - Ma)/tau - (lse_tau - Ma/tau), Ma = max(M, z_t):
                    //   KL = E_q[(u - Mu) - (z - Ma)] / tau - ln Su + (lse_tau - Ma/tau).
                    // W and Sun leave the target column out, so with c = Mu - Ma
                    //   Su E_q[(u - Mu) - (z - Ma)] = (W - c Sun) + e_t ((u_t - z_t) - c),
                    // e_t = e^((u_t - Mu)/tau): the target's part is exactly 0 when teacher
                    // and student both have their maximum there, and then
                    // ln Su = (u_t - Mu)/tau + log1p(Sun / e_t) keeps full precision;
                    // lse_tau - Ma/tau = softplus(dT) when z_t >= M, rb otherwise (below;
                    // at tau = 1 the NLL, or ln S + softplus(-d)).  No term grows with the
                    // logits' offset, so a small KL (both confident on the target) keeps
                    // its digits.
                    float kl = 0.f;
                    // tau != 1: the tempered student p^tau = softmax(z / tau) has
                    //   lse_tau = logaddexp(z_t / tau, M / tau + ln St) = mr / tau + rb
                    // with the reference point mr = M (z_t when no other column is
                    // finite) and, as for the cross-entropy, dT = (M - z_t) / tau + ln St,
                    // rb = ln St + softplus(-dT), p^tau_t = sigmoid(-dT)
                    // ln Su twice: precisely for the KL (a small KL is a difference of such
                    // logarithms), by the fast intrinsic for the teacher's gradient offset,
                    // which sits on the chain to pass C and needs no more than 1e-6
                    float mr = 0.f, rb = 0.f, ptt = 0.f, lnSu = 0.f, lnSu_g = 0.f, Wc = 0.f;
                    if (KL) {
                        lnSu_g = __logf(Su);
                        const float kappa = TAU ? p.tau_inv : 1.f;
                        const float Ma = fmaxf(M, zt);
                        const float c = (Mu == -INFINITY || Ma == -INFINITY) ? 0.f : Mu - Ma;
                        const float du = Ut - Mu;
                        const float et = ex2(du * Lt);
                        Wc = fmaf(-c, Sun, W) + ((et > 0.f) ? et * ((Ut - zt) - c) : 0.f);
                        lnSu = (et >= 0.5f) ? fmaf(du, kappa, log1pf(__fdividef(Sun, et))) : logf(Su);
                    }
                    if (TAU) {
                        const float lnSt = (St == 0.f) ? -INFINITY : logf(St);
                        const float dT = fmaf(p.tau_inv, M - zt, lnSt);
                        float E = __expf(-fabsf(dT));
                        if (fabsf(dT) > 87.0f) E = expf(-fabsf(dT));
                        const float l1p = log1pf(E);
                        const float inv = __fdividef(1.f, 1.f + E);
                        ptt = (dT > 0.f) ? E * inv : inv;
                        mr = (St == 0.f) ? zt : M;
                        rb = (St == 0.f) ? 0.f : lnSt + (fmaxf(-dT, 0.f) + l1p);
                        if (isnan(dT)) rb = dT;
                        const float lseMa = (St == 0.f || zt >= M) ? fmaxf(dT, 0.f) + l1p : rb;
                        kl = fmaf(__fdividef(Wc, Su), p.tau_inv, lseMa - lnSu);
                    } else if (KL) {
                        // lse - Ma: NLL when the target is the maximum, else ln S + softplus(-d)
                        const float lseMa = (S == 0.f || zt >= M) ? nll : lnS + sp_neg;
                        kl = __fdividef(Wc, Su) + (lseMa - lnSu);
                    }
                    const float s = s_tok;
                    // GRPO, token level: rho = exp(logp - old), L = -min(rho A, clamp(rho) A);
                    // when the unclipped branch is taken its gradient is s A rho (p - onehot)
                    float c_r = 0.f, pol = 0.f;
                    if (p.tok_adv) {
                        if (!KL && !bad) load_policy();
                        const float rho = expf(-nll - g_old);
                        const float rc = fminf(fmaxf(rho, 1.f - p.eps_lo), 1.f + p.eps_hi);
                        pol = -fminf(rho * g_adv, rc * g_adv);
                        if (rho * g_adv <= rc * g_adv) c_r = s * g_adv * rho;
                        if (isnan(rho) || isnan(g_adv)) { pol = rho + g_adv; c_r = pol; }
                    }
                    *coef = row_coef<KL, TAU>(s, p.w_ce, p.alpha, p.w_kl, lse, tg, pt, c_r, b_kl, log2_b, a_fixed,
                                              log2_a_fixed, Mu, lnSu_g, mr, rb, ptt);
                    if (rank == 0) {
                        p.ws.row_nll[r] = nll;
                        p.ws.row_lse[r] = lse;
                        p.ws.row_kl[r] = kl;
                        p.ws.row_pol[r] = pol;
                        // the teacher's statistics, for GSPO's gradient pass
                        if (KL && EARLY && p.seg_ids) {
                            reinterpret_cast<float2*>(p.ws.row_tu)[r] = make_float2(Mu, lnSu_g);
                            if (TAU) reinterpret_cast<float4*>(p.ws.row_tt)[r] = make_float4(mr, rb, ptt, 0.f);
                        }
                        if (LMLOSS_ENT_RT) {
                            // H = sum p (-log p): the target gives p_t NLL; a non-target j gives
                            // p_j (lse - z_j) with p_j = p_nt e^(z_j - M) / S and
                            // lse - z_j = ln S + softplus(-d) - (z_j - M), so
                            //   H = p_t NLL + p_nt (ln S - B/S + softplus(-d)),
                            // every term non-negative (ln S - B/S is the entropy of the
                            // non-target distribution), hence no cancellation on confident rows
                            float h = (pt > 0.f) ? pt * nll : 0.f;
                            if (S > 0.f) h = fmaf(pnt, (lnS - Bc / S) + sp_neg, h);
                            p.entropy_out[r] = h;
                        }
                        if (p.logp_out) p.logp_out[r] = -nll;
                        if (p.lse_out) p.lse_out[r] = lse;
                        if (p.kl_out) p.kl_out[r] = kl;
                    }
                }
            } else if (lane == 0 && rank == 0 && mode != kModeGrad) {
                p.ws.row_nll[r] = 0.f; p.ws.row_lse[r] = 0.f; p.ws.row_kl[r] = 0.f; p.ws.row_pol[r] = 0.f;
                if (EARLY && p.part_out) {
                    float* o = p.part_out + 4 * r;
                    o[0] = -INFINITY; o[1] = 0.f; o[2] = 0.f; o[3] = 0.f;
                }
                if (LMLOSS_ENT_RT) p.entropy_out[r] = 0.f;
                if (p.logp_out) p.logp_out[r] = 0.f;
                if (p.lse_out) p.lse_out[r] = 0.f;
                if (p.kl_out) p.kl_out[r] = 0.f;
            }
            if (lane == 0) {
                rowq[(i + depth) & 3] = next_row;
                tq[(i + depth) & 3] = next_t;
            }
        }
        __syncthreads();

        // ---- pass C: gradient of the slice, written once
        if (p.grad && mode != kModeStats) {
            unsigned char* g = static_cast<unsigned char*>(p.grad) + row_off + static_cast<size_t>(e0) * ESZ;
            if (!act) {
                for (int v = tid; v < nvec; v += NT) stg128(g + static_cast<size_t>(v) * 16, make_uint4(0, 0, 0, 0));
                if (tid == NT - 1) {
                    for (int64_t j = c0; j < e0; ++j) IO::store1(p.grad, r * p.ld + j, 0.f);
                    for (int64_t j = e1; j < c1; ++j) IO::store1(p.grad, r * p.ld + j, 0.f);
                }
                continue;
            }
            const RowCoef cf = *coef;
            if (TAU && !cf.neg && cf.b > 0.f) {
                // g_j = 2^(z_j log2e - cz) + 2^((z_j - mr) Lt - ct) - 2^((u_j - mu) Lt - cq)
                const uint64_t L2 = f2_pack(kLog2e, kLog2e);
                const uint64_t Lt2 = f2_pack(Lt, Lt);
                const uint64_t ncz = f2_pack(-cf.cz, -cf.cz);
                const uint64_t nct = f2_pack(-cf.ct, -cf.ct);
                const uint64_t ncq = f2_pack(-cf.cq, -cf.cq);
                const uint64_t nmr = f2_pack(-cf.mr, -cf.mr);
                const uint64_t nmu = f2_pack(-cf.mu, -cf.mu);
                const uint64_t neg1 = f2_pack(-1.f, -1.f);
                auto vec = [&](int v, int tcol) {
                    const uint4 q = lds128(bz + v * 16);
                    const uint4 qu = lds128(bu + v * 16);
                    float gv[VN];
#pragma unroll
                    for (int k = 0; k < VN / 2; ++k) {
                        const uint64_t xz = IO::pair(q, k);
                        float a0, a1, t0, t1, b0, b1;
                        f2_unpack(f2_fma(xz, L2, ncz), a0, a1);
                        f2_unpack(f2_fma(f2_add(xz, nmr), Lt2, nct), t0, t1);
                        f2_unpack(f2_fma(f2_add(IO::pair(qu, k), nmu), Lt2, ncq), b0, b1);
                        const uint64_t bq = f2_pack(ex2(b0), ex2(b1));
                        const uint64_t ap = f2_add(f2_pack(ex2(a0), ex2(a1)), f2_pack(ex2(t0), ex2(t1)));
                        float g0, g1;
                        f2_unpack(f2_fma(bq, neg1, ap), g0, g1);
                        if (tcol >= 0) {
                            float q0, q1;
                            f2_unpack(bq, q0, q1);
                            if (2 * k == tcol) g0 = cf.gt - q0;
                            if (2 * k + 1 == tcol) g1 = cf.gt - q1;
                        }
                        gv[2 * k] = g0;
                        gv[2 * k + 1] = g1;
                    }
                    stg128(g + static_cast<size_t>(v) * 16, IO::pack(gv));
                };
#pragma unroll 2
                for (int v = tid; v < nvec; v += NT)
                    if (v != vt) vec(v, -1);
                if (vt >= 0 && vt % NT == tid) vec(vt, kt);
            } else if (TAU) {
                // a < 0 or b <= 0: g_j = a p_j + b (p^tau_j - q_j)
#pragma unroll 2
                for (int v = tid; v < nvec; v += NT) {
                    float x[VN], y[VN], gv[VN], qv[VN];
                    IO::unpack(lds128(bz + v * 16), x);
                    IO::unpack(lds128(bu + v * 16), y);
#pragma unroll
                    for (int j = 0; j < VN; ++j) {
                        qv[j] = cf.b * ex2(fmaf(y[j] - cf.mu, Lt, -cf.luL));
                        const float ptj = ex2(fmaf(x[j] - cf.mr, Lt, -cf.ltL));
                        gv[j] = fmaf(cf.a, ex2(fmaf(x[j], kLog2e, -cf.lseL)), fmaf(cf.b, ptj, -qv[j]));
                    }
                    if (v == vt) {
#pragma unroll
                        for (int j = 0; j < VN; ++j)
                            if (j == kt) gv[j] = cf.gt - qv[j];
                    }
                    stg128(g + static_cast<size_t>(v) * 16, IO::pack(gv));
                }
            } else if (KL && cf.a > 0.f && cf.b > 0.f) {
                // g_j = 2^(z_j log2e - cz) - 2^(u_j log2e - cq): both coefficients in the exponents
                const uint64_t L2 = f2_pack(kLog2e, kLog2e);
                const uint64_t ncz = f2_pack(-cf.cz, -cf.cz);
                const uint64_t ncq = f2_pack(-cf.cq, -cf.cq);
                const uint64_t neg1 = f2_pack(-1.f, -1.f);
                auto vec = [&](int v, int tcol) {
                    const uint4 q = lds128(bz + v * 16);
                    const uint4 qu = lds128(bu + v * 16);
                    float gv[VN];
#pragma unroll
                    for (int k = 0; k < VN / 2; ++k) {
                        float a0, a1, b0, b1;
                        f2_unpack(f2_fma(IO::pair(q, k), L2, ncz), a0, a1);
                        f2_unpack(f2_fma(IO::pair(qu, k), L2, ncq), b0, b1);
                        const uint64_t bq = f2_pack(ex2(b0), ex2(b1));
                        const uint64_t ap = f2_pack(ex2(a0), ex2(a1));
                        float g0, g1;
                        f2_unpack(f2_fma(bq, neg1, ap), g0, g1);
                        if (tcol >= 0) {
                            float q0, q1;
                            f2_unpack(bq, q0, q1);
                            if (2 * k == tcol) g0 = cf.gt - q0;
                            if (2 * k + 1 == tcol) g1 = cf.gt - q1;
                        }
                        gv[2 * k] = g0;
                        gv[2 * k + 1] = g1;
                    }
                    stg128(g + static_cast<size_t>(v) * 16, IO::pack(gv));
                };
                // the target's vector out of the loop: no per-column test inside it
#pragma unroll 2
                for (int v = tid; v < nvec; v += NT)
                    if (v != vt) vec(v, -1);
                if (vt >= 0 && vt % NT == tid) vec(vt, kt);
            } else if (KL) {
#pragma unroll 2
                for (int v = tid; v < nvec; v += NT) {
                    float x[VN], y[VN], gv[VN], qv[VN];
                    IO::unpack(lds128(bz + v * 16), x);
                    IO::unpack(lds128(bu + v * 16), y);
#pragma unroll
                    for (int j = 0; j < VN; ++j) {
                        qv[j] = cf.b * ex2(fmaf(y[j], kLog2e, -cf.luL));
                        gv[j] = fmaf(cf.a, ex2(fmaf(x[j], kLog2e, -cf.lseL)), -qv[j]);
                    }
                    if (v == vt) {
#pragma unroll
                        for (int j = 0; j < VN; ++j)
                            if (j == kt) gv[j] = cf.gt - qv[j];
                    }
                    stg128(g + static_cast<size_t>(v) * 16, IO::pack(gv));
                }
            } else {
                auto body = [&](auto NEG) {
                    // g_j = (+-) 2^(z_j log2e - cz), two arguments per f32x2 FMA
                    const uint64_t L2 = f2_pack(kLog2e, kLog2e);
                    const uint64_t ncz = f2_pack(-cf.cz, -cf.cz);
#pragma unroll 2
                    for (int v = tid; v < nvec; v += NT) {
                        const uint4 q = lds128(bz + v * 16);
                        float gv[VN];
#pragma unroll
                        for (int k = 0; k < VN / 2; ++k) {
                            float a0, a1;
                            f2_unpack(f2_fma(IO::pair(q, k), L2, ncz), a0, a1);
                            gv[2 * k] = ex2(a0);
                            gv[2 * k + 1] = ex2(a1);
                        }
                        if (decltype(NEG)::value) {
#pragma unroll
                            for (int j = 0; j < VN; ++j) gv[j] = -gv[j];
                        }
                        if (v == vt) {
#pragma unroll
                            for (int j = 0; j < VN; ++j)
                                if (j == kt) gv[j] = cf.gt;
                        }
                        stg128(g + static_cast<size_t>(v) * 16, IO::pack(gv));
                    }
                };
                if (cf.neg) body(BoolConst<true>{});
                else body(BoolConst<false>{});
            }
            if (tid == NT - 1) {
                for (int pass = 0; pass < 2; ++pass) {
                    const int64_t lo = pass == 0 ? c0 : e1, hi = pass == 0 ? e0 : c1;
                    for (int64_t j = lo; j < hi; ++j) {
                        const float x = IO::load1(p.logits, r * p.ld + j);
                        float gj;
                        if (TAU) {
                            const float y = IO::load1(p.teacher, r * p.ld + j);
                            const float qj = cf.b * ex2(fmaf(y - cf.mu, Lt, -cf.luL));
                            const float ptj = ex2(fmaf(x - cf.mr, Lt, -cf.ltL));
                            gj = (j == t) ? cf.gt - qj
                                          : fmaf(cf.a, ex2(fmaf(x, kLog2e, -cf.lseL)), fmaf(cf.b, ptj, -qj));
                        } else if (KL) {
                            const float qj = cf.b * ex2(fmaf(IO::load1(p.teacher, r * p.ld + j), kLog2e, -cf.luL));
                            gj = (j == t) ? cf.gt - qj : fmaf(cf.a, ex2(fmaf(x, kLog2e, -cf.lseL)), -qj);
                        } else {
                            const float e = ex2(fmaf(x, kLog2e, -cf.cz));
                            gj = (j == t) ? cf.gt : (cf.neg ? -e : e);
                        }
                        IO::store1(p.grad, r * p.ld + j, gj);
                    }
                }
            }
        }
    }
#undef LMLOSS_ENT_RT
    grid_dep_launch();    // the reduction after this kernel may begin launching
    cluster_sync_all();   // no CTA leaves while a peer may still read its records
    // the last CTA to finish returns the row counter to zero for the next launch
    if (tid == 0) {
        __threadfence();
        if (atomicAdd(&p.ws.done[2], 1u) == gridDim.x - 1) {
            *p.ws.row_counter = 0;
            p.ws.done[2] = 0u;
        }
    }
}

}  // namespace lmloss
