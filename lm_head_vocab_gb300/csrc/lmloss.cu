// Host side of the lmloss C ABI: argument validation, workspace, launch
// planning and kernel sequencing.  Every step of the loss runs in the kernels
// of kernels.cuh; nothing here touches tensor data.
#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <new>

#include <cuda_runtime.h>

#include "../../include/lmloss.h"
#include "kernels.cuh"
#include "aux_kernels.cuh"
#include "fused_entry.cuh"

using namespace lmloss;

struct lmloss_ctx {
    int device = 0;
    int64_t max_T = 0;
    int32_t max_S = 0;
    void* ws_mem = nullptr;
    Workspace ws{};
    int cfg_cluster = 0, cfg_threads = 0, cfg_nbuf = 0;
    int timing = 0;
    static constexpr int kMaxTimed = 4096;
    cudaEvent_t* ev = nullptr;   // [2 * kMaxTimed], created on first use
    int ev_created = 0;          // pairs created
    int ev_used = 0;             // pairs recorded since timing was enabled
    lmloss_call_info info{};
    int num_sms = 0;
    int smem_optin = 0;
    // lmloss_forward_backward_host: a stream of the handle's own for the rows'
    // copies, and events: [0] the caller's stream reached the call, [1 + k]
    // chunk k has landed (created on first use)
    static constexpr int kMaxChunks = 64;
    cudaStream_t copy_stream = nullptr;
    cudaEvent_t cev[kMaxChunks + 1] = {};
    bool copy_ready = false;
};

namespace {

struct DeviceGuard {
    int prev = -1;
    bool ok = true;
    explicit DeviceGuard(int dev)
    {
        if (cudaGetDevice(&prev) != cudaSuccess) { ok = false; return; }
        if (prev != dev && cudaSetDevice(dev) != cudaSuccess) ok = false;
    }
    ~DeviceGuard()
    {
        if (prev >= 0) cudaSetDevice(prev);
    }
};

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

bool misaligned(const void* a, const void* b)
{
    return ((reinterpret_cast<uintptr_t>(a) - reinterpret_cast<uintptr_t>(b)) & 15u) != 0;
}

// need_loss: the call writes loss_out (every call but the shard passes that
// only read or write per-row data)
lmloss_status check(const lmloss_args* a, bool need_loss = true)
{
    if (!a) return LMLOSS_ERR_INVALID_ARG;
    if (a->T < 0 || a->V < 1 || a->ld < a->V) return LMLOSS_ERR_INVALID_ARG;
    if (a->dtype != LMLOSS_BF16 && a->dtype != LMLOSS_FP32) return LMLOSS_ERR_INVALID_ARG;
    if (a->reduction != LMLOSS_REDUCE_SUM && a->reduction != LMLOSS_REDUCE_TOKEN_MEAN) return LMLOSS_ERR_INVALID_ARG;
    if (need_loss && !a->loss_out) return LMLOSS_ERR_INVALID_ARG;
    const int esz = a->dtype == LMLOSS_BF16 ? 2 : 4;
    if (a->T > 0) {
        if (!a->logits || !a->targets) return LMLOSS_ERR_INVALID_ARG;
        if (reinterpret_cast<uintptr_t>(a->logits) % esz) return LMLOSS_ERR_INVALID_ARG;
        // T * ld elements must be addressable in bytes with int64
        if (a->ld > (INT64_MAX / 8) / a->T) return LMLOSS_ERR_INVALID_ARG;
    }
    if (a->reduction == LMLOSS_REDUCE_SUM && !(a->denominator > 0.0 && std::isfinite(a->denominator)))
        return LMLOSS_ERR_INVALID_ARG;
    if (!std::isfinite(a->ce_weight) || !std::isfinite(a->z_alpha)) return LMLOSS_ERR_INVALID_ARG;
    if (a->grad_out && a->T > 0 && misaligned(a->grad_out, a->logits)) return LMLOSS_ERR_INVALID_ARG;
    if (a->teacher_logits) {
        if (a->T > 0 && misaligned(a->teacher_logits, a->logits)) return LMLOSS_ERR_INVALID_ARG;
        if (!std::isfinite(a->kl_weight) || !(a->temperature > 0.f) || !std::isfinite(a->temperature))
            return LMLOSS_ERR_INVALID_ARG;
        if (a->grad_out == a->teacher_logits) return LMLOSS_ERR_INVALID_ARG;
    }
    if (a->segment_ids) {
        if (a->num_segments < 0) return LMLOSS_ERR_INVALID_ARG;
        if (a->T > 0 && !a->old_logprobs) return LMLOSS_ERR_INVALID_ARG;
        if (a->num_segments > 0 && !a->advantages) return LMLOSS_ERR_INVALID_ARG;
        if (!(a->clip_eps_low >= 0.f) || !(a->clip_eps_high >= 0.f)) return LMLOSS_ERR_INVALID_ARG;
    }
    if (a->token_advantages) {
        if (a->segment_ids) return LMLOSS_ERR_INVALID_ARG;   // one policy term per call
        if (a->T > 0 && !a->old_logprobs) return LMLOSS_ERR_INVALID_ARG;
        if (!(a->clip_eps_low >= 0.f) || !(a->clip_eps_high >= 0.f)) return LMLOSS_ERR_INVALID_ARG;
    }
    return LMLOSS_OK;
}

// ------------------------------------------------------------ launch plans
// tau: distillation at a temperature other than 1 (kl only); ent: the entropy
// output, a compile-time choice without a teacher (with one the kernel decides
// at run time)
const void* pick_fused(bool bf16, bool kl, bool tau, bool ent, int nt, bool stats)
{
    if (!kl) {
        if (ent) return bf16 ? fused_entry<true, false, false, true>(nt, stats)
                             : fused_entry<false, false, false, true>(nt, stats);
        return bf16 ? fused_entry<true, false, false, false>(nt, stats) : fused_entry<false, false, false, false>(nt, stats);
    }
    if (bf16)
        return tau ? fused_entry<true, true, true, false>(nt, stats) : fused_entry<true, true, false, false>(nt, stats);
    return tau ? fused_entry<false, true, true, false>(nt, stats) : fused_entry<false, true, false, false>(nt, stats);
}

struct FusedPlan {
    const void* fn = nullptr;
    int C = 0, NT = 0, nbuf = 0, grid = 0;
    int64_t slice = 0;
    uint32_t buf_bytes = 0;
    size_t smem = 0;
};

size_t fused_smem(int64_t V, int C, int nbuf, bool kl, int esz, int64_t* slice_out, uint32_t* buf_out)
{
    const int vn = 16 / esz;
    int64_t slice = (V + C - 1) / C;
    slice = (slice + vn - 1) / vn * vn;
    const uint32_t buf = static_cast<uint32_t>(align_up(static_cast<size_t>(slice) * esz, 128));
    if (slice_out) *slice_out = slice;
    if (buf_out) *buf_out = buf;
    return kHdrBytes + static_cast<size_t>(nbuf) * (kl ? 2 : 1) * buf;
}

// The dynamic shared-memory limit and the non-portable cluster permission are
// attributes of a kernel function on a device, shared by every handle and host
// thread.  They are raised once per (device, function) to the device's opt-in
// maximum, so a call on one handle never lowers the limit under another
// handle's launch.
lmloss_status raise_limits(const void* fn, int device, int smem_optin)
{
    constexpr int kMaxEntries = 1024;
    static std::mutex mu;
    static const void* fns[kMaxEntries];
    static int devs[kMaxEntries];
    static int n = 0;
    std::lock_guard<std::mutex> lock(mu);
    for (int i = 0; i < n; ++i)
        if (fns[i] == fn && devs[i] == device) return LMLOSS_OK;
    if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_optin) != cudaSuccess) {
        cudaGetLastError();
        return LMLOSS_ERR_CUDA;
    }
    if (cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess) {
        cudaGetLastError();
        return LMLOSS_ERR_UNSUPPORTED;
    }
    if (n < kMaxEntries) {
        fns[n] = fn;
        devs[n] = device;
        ++n;
    }
    return LMLOSS_OK;
}

lmloss_status plan_fused(lmloss_ctx* h, const lmloss_args* a, int mode, FusedPlan& P)
{
    const bool bf16 = a->dtype == LMLOSS_BF16;
    const bool kl = a->teacher_logits != nullptr;
    const int esz = bf16 ? 2 : 4;
    // Default shape, from sweeps on GB300: one staged row per CTA; the
    // smallest cluster whose slice (logits, plus teacher) fits in 56 KB (112 KB
    // with a teacher), so that four (two) CTAs share an SM; and about 110
    // elements per thread (55 for the gradient pass with a teacher, whose two
    // CTAs per SM need more warps to hide latency), rounded to 128, 256 or 512
    // threads.
    int nbuf = h->cfg_nbuf ? h->cfg_nbuf : 1;
    int C = h->cfg_cluster;
    if (!C) {
        const int64_t row_bytes = a->V * esz * (kl ? 2 : 1);
        const int64_t budget = kl ? 112 * 1024 : 56 * 1024;
        int64_t c = (row_bytes + budget - 1) / budget;
        C = static_cast<int>(c < 1 ? 1 : (c > 16 ? 16 : c));
    }
    int NT = h->cfg_threads;
    if (!NT) {
        const double per_thread = static_cast<double>((a->V + C - 1) / C) / (kl && mode != kModeStats ? 55.0 : 110.0);
        NT = per_thread < 181.0 ? 128 : (per_thread < 362.0 ? 256 : 512);
    }
    if (a->T >= (int64_t(1) << 30)) return LMLOSS_ERR_UNSUPPORTED;   // row indices are 32-bit in the kernel
    if (C < 1 || C > 16 || (nbuf != 1 && nbuf != 2)) return LMLOSS_ERR_UNSUPPORTED;
    P.fn = pick_fused(bf16, kl, kl && a->temperature != 1.0f, a->entropy_out != nullptr, NT, mode == kModeStats);
    if (!P.fn) return LMLOSS_ERR_UNSUPPORTED;
    P.C = C;
    P.NT = NT;
    P.nbuf = nbuf;
    P.smem = fused_smem(a->V, C, nbuf, kl, esz, &P.slice, &P.buf_bytes);
    // a row whose slices do not fit one CTA's shared memory even at 16 CTAs a row
    if (P.smem > static_cast<size_t>(h->smem_optin)) return LMLOSS_ERR_UNSUPPORTED;
    lmloss_status st = raise_limits(P.fn, h->device, h->smem_optin);
    if (st != LMLOSS_OK) return st;
    cudaLaunchConfig_t cfg{};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = C;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3(static_cast<unsigned>(C * h->num_sms));
    cfg.blockDim = dim3(static_cast<unsigned>(NT));
    cfg.dynamicSmemBytes = P.smem;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int nclusters = 0;
    if (cudaOccupancyMaxActiveClusters(&nclusters, P.fn, &cfg) != cudaSuccess) {
        cudaGetLastError();
        return LMLOSS_ERR_UNSUPPORTED;
    }
    if (nclusters < 1) return LMLOSS_ERR_UNSUPPORTED;
    int64_t want = a->T < nclusters ? a->T : nclusters;
    if (want < 1) want = 1;
    P.grid = static_cast<int>(want) * C;
    return LMLOSS_OK;
}

void fill_params(const lmloss_ctx* h, const lmloss_args* a, CallParams& p)
{
    const bool kl = a->teacher_logits != nullptr;
    const bool gspo = a->segment_ids != nullptr;
    p.logits = a->logits;
    p.teacher = a->teacher_logits;
    p.grad = a->grad_out;
    p.targets = a->targets;
    p.mask = a->loss_mask;
    p.T = a->T;
    p.V = a->V;
    p.ld = a->ld;
    p.w_ce = a->ce_weight;
    p.alpha = a->z_alpha;
    p.w_kl = kl ? a->kl_weight : 0.f;
    // 1 / tau and log2(e) / tau, each rounded once
    p.tau_inv = kl ? static_cast<float>(1.0 / static_cast<double>(a->temperature)) : 1.f;
    p.tau_l2 = kl ? static_cast<float>(1.4426950408889634 / static_cast<double>(a->temperature)) : kLog2e;
    p.reduction = a->reduction;
    p.inv_denominator = a->reduction == LMLOSS_REDUCE_SUM ? 1.0 / a->denominator : 0.0;
    p.seg_ids = a->segment_ids;
    p.num_segments = gspo ? a->num_segments : 0;
    p.adv = a->advantages;
    p.old_logp = a->old_logprobs;
    p.eps_lo = a->clip_eps_low;
    p.eps_hi = a->clip_eps_high;
    p.loss_out = a->loss_out;
    p.logp_out = a->logp_out;
    p.lse_out = a->lse_out;
    p.kl_out = a->kl_out;
    p.count_out = a->count_out;
    p.seg_count_out = a->seg_count_out;
    p.seg_ratio_out = a->seg_ratio_out;
    p.seg_flag_out = a->seg_flag_out;
    p.seg_loss_out = a->seg_loss_out;
    p.tok_adv = a->token_advantages;
    p.entropy_out = a->entropy_out;
    p.ws = h->ws;
    p.col0 = 0;
    p.v_total = a->V;
    p.part_out = nullptr;
}

// The parameters of rows [r0, r1) as a call of their own: every row-indexed
// pointer (inputs, per-row outputs and the workspace's per-row results) moved
// to row r0, so each row keeps its place; the token scale still comes from the
// whole call's count.
CallParams chunk_params(const CallParams& p, const lmloss_args* a, int64_t r0, int64_t r1)
{
    CallParams c = p;
    const size_t off = static_cast<size_t>(r0) * static_cast<size_t>(a->ld) * (a->dtype == LMLOSS_BF16 ? 2u : 4u);
    c.logits = static_cast<const unsigned char*>(p.logits) + off;
    if (p.teacher) c.teacher = static_cast<const unsigned char*>(p.teacher) + off;
    if (p.grad) c.grad = static_cast<unsigned char*>(p.grad) + off;
    c.targets = p.targets + r0;
    if (p.mask) c.mask = p.mask + r0;
    c.T = r1 - r0;
    if (p.logp_out) c.logp_out = p.logp_out + r0;
    if (p.lse_out) c.lse_out = p.lse_out + r0;
    if (p.kl_out) c.kl_out = p.kl_out + r0;
    if (p.entropy_out) c.entropy_out = p.entropy_out + r0;
    if (p.tok_adv) c.tok_adv = p.tok_adv + r0;
    if (p.old_logp) c.old_logp = p.old_logp + r0;
    if (p.seg_ids) c.seg_ids = p.seg_ids + r0;
    c.ws.row_nll = p.ws.row_nll + r0;
    c.ws.row_lse = p.ws.row_lse + r0;
    c.ws.row_kl = p.ws.row_kl + r0;
    c.ws.row_pol = p.ws.row_pol + r0;
    c.ws.row_tu = p.ws.row_tu + 2 * r0;
    c.ws.row_tt = p.ws.row_tt + 4 * r0;
    return c;
}

lmloss_status launch_err()
{
    return cudaGetLastError() == cudaSuccess ? LMLOSS_OK : LMLOSS_ERR_CUDA;
}

// The loss reduction, launched so that it may start while the staged-row
// kernel before it finishes (it waits for that kernel's writes first).
lmloss_status launch_reduce(const CallParams& p, int blocks, cudaStream_t stream)
{
    cudaLaunchConfig_t cfg{};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.gridDim = dim3(static_cast<unsigned>(blocks));
    cfg.blockDim = dim3(256);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    CallParams q = p;
    void* kargs[] = {&q};
    if (cudaLaunchKernelExC(&cfg, reinterpret_cast<const void*>(reduce_kernel), kargs) != cudaSuccess) {
        cudaGetLastError();
        return LMLOSS_ERR_CUDA;
    }
    return LMLOSS_OK;
}

// Plan and launch the staged-row kernel in one of its modes.
lmloss_status launch_fused(lmloss_ctx* h, const lmloss_args* a, CallParams& p, int mode, cudaStream_t stream,
                           lmloss_call_info& info)
{
    FusedPlan P;
    lmloss_status st = plan_fused(h, a, mode, P);
    if (st != LMLOSS_OK) return st;
    p.mode = mode;
    p.cluster = P.C;
    p.slice = P.slice;
    p.nbuf = P.nbuf;
    p.buf_bytes = P.buf_bytes;
    cudaLaunchConfig_t cfg{};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = P.C;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3(static_cast<unsigned>(P.grid));
    cfg.blockDim = dim3(static_cast<unsigned>(P.NT));
    cfg.dynamicSmemBytes = P.smem;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    void* kargs[] = {&p};
    if (cudaLaunchKernelExC(&cfg, P.fn, kargs) != cudaSuccess) {
        cudaGetLastError();
        return LMLOSS_ERR_CUDA;
    }
    info.launches += 1;
    info.cluster = P.C;
    info.threads = P.NT;
    info.nbuf = P.nbuf;
    info.grid = P.grid;
    info.smem_bytes = static_cast<int32_t>(P.smem);
    return LMLOSS_OK;
}

}  // namespace

extern "C" {

const char* lmloss_status_string(lmloss_status s)
{
    switch (s) {
    case LMLOSS_OK: return "ok";
    case LMLOSS_ERR_INVALID_ARG: return "invalid argument";
    case LMLOSS_ERR_UNSUPPORTED: return "unsupported configuration";
    case LMLOSS_ERR_CUDA: return "CUDA runtime error";
    case LMLOSS_ERR_BAD_TARGET: return "target outside [0, V) and not ignore_index";
    case LMLOSS_ERR_BAD_SEGMENT: return "segment id outside [0, num_segments)";
    case LMLOSS_ERR_RANGE: return "GSPO log-ratio sum out of range";
    case LMLOSS_ERR_TIMEOUT: return "bounded wait on a copy expired";
    }
    return "unknown status";
}

lmloss_status lmloss_check_args(const lmloss_args* args) { return check(args); }

lmloss_status lmloss_create(lmloss_handle* handle, int device, int64_t max_T, int32_t max_segments)
{
    if (!handle || max_T < 0 || max_segments < 0) return LMLOSS_ERR_INVALID_ARG;
    *handle = nullptr;
    DeviceGuard g(device);
    if (!g.ok) return LMLOSS_ERR_CUDA;
    lmloss_ctx* h = new (std::nothrow) lmloss_ctx();
    if (!h) return LMLOSS_ERR_CUDA;
    h->device = device;
    h->max_T = max_T;
    h->max_S = max_segments;
    if (cudaDeviceGetAttribute(&h->num_sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess ||
        cudaDeviceGetAttribute(&h->smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, device) != cudaSuccess) {
        delete h;
        return LMLOSS_ERR_CUDA;
    }
    const size_t T = static_cast<size_t>(max_T > 0 ? max_T : 1);
    const size_t S = static_cast<size_t>(max_segments > 0 ? max_segments : 1);
    size_t off = 0;
    auto take = [&](size_t bytes) { size_t o = off; off = align_up(off + bytes, 256); return o; };
    const size_t o_nll = take(4 * T), o_lse = take(4 * T), o_kl = take(4 * T), o_pol = take(4 * T);
    const size_t o_tu = take(8 * T), o_tt = take(16 * T);
    const size_t o_scal = take(64);
    const size_t o_sn = take(4 * S), o_dq = take(8 * S), o_aq = take(8 * S), o_nf = take(12 * S), o_coef = take(4 * S);
    const size_t o_ctr = take(16);
    const size_t o_cnt = take(8 * kRedBlocks), o_red = take(32 * kRedBlocks), o_done = take(16);
    const size_t o_err = take(16);
    if (cudaMalloc(&h->ws_mem, off) != cudaSuccess) {
        delete h;
        return LMLOSS_ERR_CUDA;
    }
    char* base = static_cast<char*>(h->ws_mem);
    h->ws.row_nll = reinterpret_cast<float*>(base + o_nll);
    h->ws.row_lse = reinterpret_cast<float*>(base + o_lse);
    h->ws.row_kl = reinterpret_cast<float*>(base + o_kl);
    h->ws.row_pol = reinterpret_cast<float*>(base + o_pol);
    h->ws.row_tu = reinterpret_cast<float*>(base + o_tu);
    h->ws.row_tt = reinterpret_cast<float*>(base + o_tt);
    h->ws.n_active = reinterpret_cast<int64_t*>(base + o_scal);
    h->ws.n_nonempty = reinterpret_cast<int64_t*>(base + o_scal + 8);
    h->ws.gspo_sum = reinterpret_cast<double*>(base + o_scal + 16);
    h->ws.s_seg = reinterpret_cast<double*>(base + o_scal + 24);
    h->ws.seg_n = reinterpret_cast<int*>(base + o_sn);
    h->ws.seg_dq = reinterpret_cast<unsigned long long*>(base + o_dq);
    h->ws.seg_absq = reinterpret_cast<unsigned long long*>(base + o_aq);
    h->ws.seg_nonfinite = reinterpret_cast<int*>(base + o_nf);
    h->ws.seg_coef = reinterpret_cast<float*>(base + o_coef);
    h->ws.row_counter = reinterpret_cast<int*>(base + o_ctr);
    h->ws.cnt_part = reinterpret_cast<long long*>(base + o_cnt);
    h->ws.red_part = reinterpret_cast<double*>(base + o_red);
    h->ws.done = reinterpret_cast<unsigned*>(base + o_done);
    h->ws.err = reinterpret_cast<int*>(base + o_err);
    h->ev = static_cast<cudaEvent_t*>(std::calloc(2 * lmloss_ctx::kMaxTimed, sizeof(cudaEvent_t)));
    if (!h->ev || cudaMemset(h->ws_mem, 0, off) != cudaSuccess) {
        std::free(h->ev);
        cudaFree(h->ws_mem);
        delete h;
        return LMLOSS_ERR_CUDA;
    }
    *handle = h;
    return LMLOSS_OK;
}

lmloss_status lmloss_destroy(lmloss_handle h)
{
    if (!h) return LMLOSS_ERR_INVALID_ARG;
    DeviceGuard g(h->device);
    cudaDeviceSynchronize();
    if (h->copy_ready) {
        cudaStreamDestroy(h->copy_stream);
        for (cudaEvent_t e : h->cev) cudaEventDestroy(e);
    }
    for (int i = 0; i < 2 * h->ev_created; ++i) cudaEventDestroy(h->ev[i]);
    std::free(h->ev);
    cudaError_t e = cudaFree(h->ws_mem);
    delete h;
    return e == cudaSuccess ? LMLOSS_OK : LMLOSS_ERR_CUDA;
}

lmloss_status lmloss_set_launch_config(lmloss_handle h, int cluster, int threads, int nbuf)
{
    if (!h) return LMLOSS_ERR_INVALID_ARG;
    if (cluster < 0 || cluster > 16) return LMLOSS_ERR_INVALID_ARG;
    if (threads != 0 && threads != 128 && threads != 256 && threads != 512 && threads != 1024)
        return LMLOSS_ERR_INVALID_ARG;
    if (nbuf < 0 || nbuf > 2) return LMLOSS_ERR_INVALID_ARG;
    h->cfg_cluster = cluster;
    h->cfg_threads = threads;
    h->cfg_nbuf = nbuf;
    return LMLOSS_OK;
}

lmloss_status lmloss_set_timing(lmloss_handle h, int enable)
{
    if (!h) return LMLOSS_ERR_INVALID_ARG;
    h->timing = enable ? 1 : 0;
    h->ev_used = 0;
    return LMLOSS_OK;
}

lmloss_status lmloss_get_timing(lmloss_handle h, float* total_ms, int32_t* calls)
{
    if (!h || !total_ms) return LMLOSS_ERR_INVALID_ARG;
    DeviceGuard g(h->device);
    float sum = 0.f;
    for (int i = 0; i < h->ev_used; ++i) {
        float ms = 0.f;
        if (cudaEventSynchronize(h->ev[2 * i + 1]) != cudaSuccess) return LMLOSS_ERR_CUDA;
        if (cudaEventElapsedTime(&ms, h->ev[2 * i], h->ev[2 * i + 1]) != cudaSuccess) return LMLOSS_ERR_CUDA;
        sum += ms;
    }
    *total_ms = sum;
    if (calls) *calls = h->ev_used;
    return LMLOSS_OK;
}

lmloss_status lmloss_get_call_info(lmloss_handle h, lmloss_call_info* info)
{
    if (!h || !info) return LMLOSS_ERR_INVALID_ARG;
    *info = h->info;
    return LMLOSS_OK;
}

lmloss_status lmloss_get_device_error(lmloss_handle h)
{
    if (!h) return LMLOSS_ERR_INVALID_ARG;
    DeviceGuard g(h->device);
    if (!g.ok || cudaDeviceSynchronize() != cudaSuccess) return LMLOSS_ERR_CUDA;
    int code = 0;
    if (cudaMemcpy(&code, h->ws.err, sizeof code, cudaMemcpyDeviceToHost) != cudaSuccess) return LMLOSS_ERR_CUDA;
    if (cudaMemset(h->ws.err, 0, sizeof code) != cudaSuccess) return LMLOSS_ERR_CUDA;
    return static_cast<lmloss_status>(code);
}

lmloss_status lmloss_selftest_bounded_wait(lmloss_handle h, long long limit_cycles)
{
    if (!h || limit_cycles < 0) return LMLOSS_ERR_INVALID_ARG;
    DeviceGuard g(h->device);
    if (!g.ok) return LMLOSS_ERR_CUDA;
    // the handle's error word doubles as the result slot (it is read back and cleared here)
    if (cudaMemset(h->ws.err, 0, sizeof(int)) != cudaSuccess) return LMLOSS_ERR_CUDA;
    wait_selftest_kernel<<<1, 32>>>(limit_cycles, h->ws.err);
    if (cudaGetLastError() != cudaSuccess || cudaDeviceSynchronize() != cudaSuccess) return LMLOSS_ERR_CUDA;
    int code = 0;
    if (cudaMemcpy(&code, h->ws.err, sizeof code, cudaMemcpyDeviceToHost) != cudaSuccess) return LMLOSS_ERR_CUDA;
    if (cudaMemset(h->ws.err, 0, sizeof code) != cudaSuccess) return LMLOSS_ERR_CUDA;
    return static_cast<lmloss_status>(code);
}

lmloss_status lmloss_forward_backward(lmloss_handle h, const lmloss_args* a, cudaStream_t stream)
{
    if (!h) return LMLOSS_ERR_INVALID_ARG;
    lmloss_status st = check(a);
    if (st != LMLOSS_OK) return st;
    if (a->T > h->max_T) return LMLOSS_ERR_INVALID_ARG;
    if (a->segment_ids && a->num_segments > h->max_S) return LMLOSS_ERR_INVALID_ARG;
    DeviceGuard g(h->device);
    if (!g.ok) return LMLOSS_ERR_CUDA;

    const bool gspo = a->segment_ids != nullptr;

    CallParams p{};
    fill_params(h, a, p);

    lmloss_call_info info{};

    // count / reduce: one block per 64 rows, at most kRedBlocks, at least one
    int64_t rb = (a->T + 63) / 64;
    if (rb > kRedBlocks) rb = kRedBlocks;
    const int red_blocks = rb < 1 ? 1 : static_cast<int>(rb);
    // The count gives the token mean its scale before any gradient is written,
    // and clears the GSPO accumulators.  Under SUM without GSPO nothing needs
    // it: the staged-row kernel flags bad targets and leaves its row counter at
    // zero, and the reduction counts the active rows itself.
    if (gspo || a->reduction == LMLOSS_REDUCE_TOKEN_MEAN) {
        count_kernel<<<red_blocks, 256, 0, stream>>>(p);
        if ((st = launch_err()) != LMLOSS_OK) return st;
        info.launches = 1;
    }

    int ev_slot = -1;
    if (h->timing && h->ev_used < lmloss_ctx::kMaxTimed) {
        ev_slot = h->ev_used;
        if (ev_slot >= h->ev_created) {
            if (cudaEventCreate(&h->ev[2 * ev_slot]) != cudaSuccess ||
                cudaEventCreate(&h->ev[2 * ev_slot + 1]) != cudaSuccess)
                return LMLOSS_ERR_CUDA;
            h->ev_created = ev_slot + 1;
        }
        cudaEventRecord(h->ev[2 * ev_slot], stream);
    }
    if (a->T > 0) {
        if (!gspo && a->grad_out) {
            // one read of the logits, one write of the gradient
            if ((st = launch_fused(h, a, p, kModeFused, stream, info)) != LMLOSS_OK) return st;
            info.path = 0;
        } else {
            // statistics pass (forward only, or the first pass of GSPO)
            if ((st = launch_fused(h, a, p, kModeStats, stream, info)) != LMLOSS_OK) return st;
            info.path = gspo ? 2 : 1;
            if (gspo) {
                const int tg = 256;
                int64_t gb = (a->T + tg - 1) / tg;
                if (gb > 4LL * h->num_sms) gb = 4LL * h->num_sms;
                seam_accum_kernel<<<static_cast<unsigned>(gb), tg, 0, stream>>>(p);
                if ((st = launch_err()) != LMLOSS_OK) return st;
                seam_finish_kernel<<<1, 1024, 0, stream>>>(p);
                if ((st = launch_err()) != LMLOSS_OK) return st;
                info.launches += 2;
                // the seam has seen every row: the gradient pass reads the logits again
                if (a->grad_out && (st = launch_fused(h, a, p, kModeGrad, stream, info)) != LMLOSS_OK) return st;
            }
        }
    }
    if (ev_slot >= 0) {
        cudaEventRecord(h->ev[2 * ev_slot + 1], stream);
        h->ev_used = ev_slot + 1;
    }
    if ((st = launch_reduce(p, red_blocks, stream)) != LMLOSS_OK) return st;
    info.launches += 1;
    h->info = info;
    return LMLOSS_OK;
}

lmloss_status lmloss_forward_backward_host(lmloss_handle h, const lmloss_args* a, const void* host_logits,
                                           const void* host_teacher, int64_t chunk_rows, cudaStream_t stream)
{
    if (!h) return LMLOSS_ERR_INVALID_ARG;
    lmloss_status st = check(a);
    if (st != LMLOSS_OK) return st;
    if (a->T > h->max_T || chunk_rows < 0) return LMLOSS_ERR_INVALID_ARG;
    if (a->T > 0 && !host_logits) return LMLOSS_ERR_INVALID_ARG;
    if ((host_teacher != nullptr) != (a->teacher_logits != nullptr)) return LMLOSS_ERR_INVALID_ARG;
    if (a->segment_ids && a->num_segments > h->max_S) return LMLOSS_ERR_INVALID_ARG;
    const bool gspo = a->segment_ids != nullptr;
    DeviceGuard g(h->device);
    if (!g.ok) return LMLOSS_ERR_CUDA;
    if (!h->copy_ready) {
        // all or nothing: what was created is destroyed again if any creation fails
        cudaStream_t cs = nullptr;
        cudaEvent_t ev[lmloss_ctx::kMaxChunks + 1] = {};
        int made = 0;
        bool ok = cudaStreamCreateWithFlags(&cs, cudaStreamNonBlocking) == cudaSuccess;
        for (; ok && made < lmloss_ctx::kMaxChunks + 1; ++made)
            ok = cudaEventCreateWithFlags(&ev[made], cudaEventDisableTiming) == cudaSuccess;
        if (!ok) {
            for (int i = 0; i < made; ++i)
                if (ev[i]) cudaEventDestroy(ev[i]);
            if (cs) cudaStreamDestroy(cs);
            cudaGetLastError();
            return LMLOSS_ERR_CUDA;
        }
        h->copy_stream = cs;
        for (int i = 0; i <= lmloss_ctx::kMaxChunks; ++i) h->cev[i] = ev[i];
        h->copy_ready = true;
    }

    CallParams p{};
    fill_params(h, a, p);
    lmloss_call_info info{};
    int64_t rb = (a->T + 63) / 64;
    if (rb > kRedBlocks) rb = kRedBlocks;
    const int red_blocks = rb < 1 ? 1 : static_cast<int>(rb);
    // the token mean's count over every row, before any chunk's gradient (it also
    // clears GSPO's segment accumulators)
    if (gspo || a->reduction == LMLOSS_REDUCE_TOKEN_MEAN) {
        count_kernel<<<red_blocks, 256, 0, stream>>>(p);
        if ((st = launch_err()) != LMLOSS_OK) return st;
        info.launches = 1;
    }
    const int64_t T = a->T;
    if (T > 0) {
        // chunks: 8 by default, at most kMaxChunks
        int64_t rows = chunk_rows > 0 ? chunk_rows : (T + 7) / 8;
        if ((T + rows - 1) / rows > lmloss_ctx::kMaxChunks) rows = (T + lmloss_ctx::kMaxChunks - 1) / lmloss_ctx::kMaxChunks;
        const int64_t nchunks = (T + rows - 1) / rows;
        const size_t esz = a->dtype == LMLOSS_BF16 ? 2u : 4u;
        const size_t row_bytes = static_cast<size_t>(a->ld) * esz;
        // the copies wait for the caller's earlier work on its stream (which may
        // still read or write these buffers), then go out back to back
        if (cudaEventRecord(h->cev[0], stream) != cudaSuccess ||
            cudaStreamWaitEvent(h->copy_stream, h->cev[0], 0) != cudaSuccess)
            return LMLOSS_ERR_CUDA;
        for (int64_t k = 0; k < nchunks; ++k) {
            const int64_t r0 = k * rows, r1 = std::min(T, r0 + rows);
            // rows r0 .. r1 - 1: every column of the full rows, the last row's V
            const size_t off = static_cast<size_t>(r0) * row_bytes;
            const size_t bytes = static_cast<size_t>(r1 - r0 - 1) * row_bytes + static_cast<size_t>(a->V) * esz;
            if (cudaMemcpyAsync(static_cast<unsigned char*>(const_cast<void*>(a->logits)) + off,
                                static_cast<const unsigned char*>(host_logits) + off, bytes, cudaMemcpyHostToDevice,
                                h->copy_stream) != cudaSuccess)
                return LMLOSS_ERR_CUDA;
            if (host_teacher &&
                cudaMemcpyAsync(static_cast<unsigned char*>(const_cast<void*>(a->teacher_logits)) + off,
                                static_cast<const unsigned char*>(host_teacher) + off, bytes, cudaMemcpyHostToDevice,
                                h->copy_stream) != cudaSuccess)
                return LMLOSS_ERR_CUDA;
            if (cudaEventRecord(h->cev[1 + k], h->copy_stream) != cudaSuccess) return LMLOSS_ERR_CUDA;
        }
        // each chunk's staged-row kernel as soon as its rows have landed: the
        // kernels run under the copies of the chunks after them.  With GSPO that
        // is the statistics pass; the seam and the gradient pass follow once
        // every row is in, as in the regular call.
        const int mode = (a->grad_out && !gspo) ? kModeFused : kModeStats;
        for (int64_t k = 0; k < nchunks; ++k) {
            const int64_t r0 = k * rows, r1 = std::min(T, r0 + rows);
            if (cudaStreamWaitEvent(stream, h->cev[1 + k], 0) != cudaSuccess) return LMLOSS_ERR_CUDA;
            lmloss_args ac = *a;
            ac.T = r1 - r0;
            CallParams pc = chunk_params(p, a, r0, r1);
            if ((st = launch_fused(h, &ac, pc, mode, stream, info)) != LMLOSS_OK) return st;
        }
        info.path = gspo ? 2 : (a->grad_out ? 0 : 1);
        if (gspo) {
            const int tg = 256;
            int64_t gb = (T + tg - 1) / tg;
            if (gb > 4LL * h->num_sms) gb = 4LL * h->num_sms;
            seam_accum_kernel<<<static_cast<unsigned>(gb), tg, 0, stream>>>(p);
            if ((st = launch_err()) != LMLOSS_OK) return st;
            seam_finish_kernel<<<1, 1024, 0, stream>>>(p);
            if ((st = launch_err()) != LMLOSS_OK) return st;
            info.launches += 2;
            if (a->grad_out && (st = launch_fused(h, a, p, kModeGrad, stream, info)) != LMLOSS_OK) return st;
        }
    }
    if ((st = launch_reduce(p, red_blocks, stream)) != LMLOSS_OK) return st;
    info.launches += 1;
    h->info = info;
    return LMLOSS_OK;
}

// ------------------------------------------------- vocabulary-split rows
// Arguments of a shard call: cross-entropy and z-loss only.
static lmloss_status check_shard(const lmloss_args* a, int64_t v0, int64_t V_total)
{
    if (!a) return LMLOSS_ERR_INVALID_ARG;
    if (a->teacher_logits || a->segment_ids || a->token_advantages || a->entropy_out || a->kl_out)
        return LMLOSS_ERR_UNSUPPORTED;
    if (v0 < 0 || V_total < 1 || a->V < 1 || v0 > V_total - a->V) return LMLOSS_ERR_INVALID_ARG;
    if (V_total > (int64_t(1) << 31) - 8) return LMLOSS_ERR_UNSUPPORTED;   // targets as int in the kernel
    return LMLOSS_OK;
}

static lmloss_status shard_prologue(lmloss_handle h, const lmloss_args* a, CallParams& p, int64_t v0, int64_t V_total,
                             cudaStream_t stream)
{
    fill_params(h, a, p);
    p.col0 = v0;
    p.v_total = V_total;
    int64_t rb = (a->T + 63) / 64;
    if (rb > kRedBlocks) rb = kRedBlocks;
    // the count gives the token scale, checks targets against the whole vocabulary
    // and resets the row counter of the fused kernel
    count_kernel<<<rb < 1 ? 1 : static_cast<unsigned>(rb), 256, 0, stream>>>(p);
    return launch_err();
}

lmloss_status lmloss_shard_stats(lmloss_handle h, const lmloss_args* a, int64_t v0, int64_t V_total,
                                 float* part_out, cudaStream_t stream)
{
    if (!h) return LMLOSS_ERR_INVALID_ARG;
    lmloss_status st = check_shard(a, v0, V_total);
    if (st != LMLOSS_OK) return st;
    lmloss_args b = *a;
    b.grad_out = nullptr;
    if ((st = check(&b, false)) != LMLOSS_OK) return st;
    if (a->T > h->max_T || (a->T > 0 && !part_out)) return LMLOSS_ERR_INVALID_ARG;
    DeviceGuard g(h->device);
    if (!g.ok) return LMLOSS_ERR_CUDA;
    CallParams p{};
    if ((st = shard_prologue(h, &b, p, v0, V_total, stream)) != LMLOSS_OK) return st;
    p.loss_out = nullptr;
    p.logp_out = p.lse_out = nullptr;
    p.part_out = part_out;
    lmloss_call_info info{};
    info.launches = 1;
    if (a->T > 0 && (st = launch_fused(h, &b, p, kModeStats, stream, info)) != LMLOSS_OK) return st;
    info.path = 3;
    h->info = info;
    return LMLOSS_OK;
}

lmloss_status lmloss_shard_merge(lmloss_handle h, const lmloss_args* a, const float* const* parts, int32_t K,
                                 cudaStream_t stream)
{
    if (!h || !a) return LMLOSS_ERR_INVALID_ARG;
    lmloss_status st = check_shard(a, 0, a->V);
    if (st != LMLOSS_OK) return st;
    if (K < 1 || K > kMaxShards || !parts) return LMLOSS_ERR_INVALID_ARG;
    if (a->T < 0 || a->T > h->max_T || !a->loss_out) return LMLOSS_ERR_INVALID_ARG;
    if (a->T > 0 && !a->targets) return LMLOSS_ERR_INVALID_ARG;
    if (a->reduction != LMLOSS_REDUCE_SUM && a->reduction != LMLOSS_REDUCE_TOKEN_MEAN) return LMLOSS_ERR_INVALID_ARG;
    if (a->reduction == LMLOSS_REDUCE_SUM && !(a->denominator > 0.0 && std::isfinite(a->denominator)))
        return LMLOSS_ERR_INVALID_ARG;
    if (!std::isfinite(a->ce_weight) || !std::isfinite(a->z_alpha)) return LMLOSS_ERR_INVALID_ARG;
    ShardParts sp{};
    sp.K = K;
    for (int k = 0; k < K; ++k) {
        if (a->T > 0 && !parts[k]) return LMLOSS_ERR_INVALID_ARG;
        sp.part[k] = parts[k];
    }
    DeviceGuard g(h->device);
    if (!g.ok) return LMLOSS_ERR_CUDA;
    CallParams p{};
    if ((st = shard_prologue(h, a, p, 0, a->V, stream)) != LMLOSS_OK) return st;
    lmloss_call_info info{};
    info.launches = 1;
    if (a->T > 0) {
        int64_t gb = (a->T + 255) / 256;
        if (gb > 4LL * h->num_sms) gb = 4LL * h->num_sms;
        shard_merge_kernel<<<static_cast<unsigned>(gb), 256, 0, stream>>>(p, sp);
        if ((st = launch_err()) != LMLOSS_OK) return st;
        info.launches += 1;
    }
    int64_t rb = (a->T + 63) / 64;
    if (rb > kRedBlocks) rb = kRedBlocks;
    reduce_kernel<<<rb < 1 ? 1 : static_cast<unsigned>(rb), 256, 0, stream>>>(p);
    if ((st = launch_err()) != LMLOSS_OK) return st;
    info.launches += 1;
    info.path = 3;
    h->info = info;
    return LMLOSS_OK;
}

lmloss_status lmloss_shard_grad(lmloss_handle h, const lmloss_args* a, int64_t v0, int64_t V_total,
                                cudaStream_t stream)
{
    if (!h) return LMLOSS_ERR_INVALID_ARG;
    lmloss_status st = check_shard(a, v0, V_total);
    if (st != LMLOSS_OK) return st;
    const lmloss_args b = *a;
    if ((st = check(&b, false)) != LMLOSS_OK) return st;
    if (a->T > h->max_T || (a->T > 0 && !a->grad_out)) return LMLOSS_ERR_INVALID_ARG;
    DeviceGuard g(h->device);
    if (!g.ok) return LMLOSS_ERR_CUDA;
    CallParams p{};
    if ((st = shard_prologue(h, &b, p, v0, V_total, stream)) != LMLOSS_OK) return st;
    p.loss_out = nullptr;
    p.logp_out = p.lse_out = nullptr;
    lmloss_call_info info{};
    info.launches = 1;
    if (a->T > 0 && (st = launch_fused(h, &b, p, kModeGrad, stream, info)) != LMLOSS_OK) return st;
    info.path = 3;
    h->info = info;
    return LMLOSS_OK;
}

}  // extern "C"

// ===========================================================================
// Allocation-free variant of lmloss_forward_backward.
//
// Some callers may not allocate device memory once they are running, for
// example an inference-engine plugin whose enqueue step must not allocate, or
// a service that plans every byte of device memory at start-up (cudaMalloc can
// synchronise the device and can fail under memory pressure).  This entry
// point takes no handle: its workspace is the fixed array below, which every
// GPU that loads this library holds until the process exits.
// ===========================================================================
namespace {

constexpr int64_t kNoAllocMaxT = LMLOSS_NOALLOC_MAX_T;
constexpr int64_t kNoAllocMaxS = LMLOSS_NOALLOC_MAX_SEGMENTS;

constexpr size_t na_align(size_t x) { return (x + 255) / 256 * 256; }

// Byte offsets of the workspace pieces inside the array.
struct NoAllocLayout {
    static constexpr size_t nll = 0;
    static constexpr size_t lse = nll + na_align(4 * kNoAllocMaxT);
    static constexpr size_t kl = lse + na_align(4 * kNoAllocMaxT);
    static constexpr size_t pol = kl + na_align(4 * kNoAllocMaxT);
    static constexpr size_t tu = pol + na_align(4 * kNoAllocMaxT);
    static constexpr size_t tt = tu + na_align(8 * kNoAllocMaxT);
    static constexpr size_t scal = tt + na_align(16 * kNoAllocMaxT);
    static constexpr size_t seg_n = scal + na_align(64);
    static constexpr size_t seg_dq = seg_n + na_align(4 * kNoAllocMaxS);
    static constexpr size_t seg_absq = seg_dq + na_align(8 * kNoAllocMaxS);
    static constexpr size_t seg_nf = seg_absq + na_align(8 * kNoAllocMaxS);
    static constexpr size_t seg_coef = seg_nf + na_align(12 * kNoAllocMaxS);
    static constexpr size_t counter = seg_coef + na_align(4 * kNoAllocMaxS);
    static constexpr size_t cnt_part = counter + na_align(16);
    static constexpr size_t red_part = cnt_part + na_align(8 * kRedBlocks);
    static constexpr size_t done = red_part + na_align(32 * kRedBlocks);
    static constexpr size_t err = done + na_align(16);
    static constexpr size_t total = err + na_align(16);
};

// The workspace itself (about 1.2 MB).  The set-up below clears it once per
// device, so the block counters that must start every call at zero do; the
// kernels return those counters to zero at the end of each call and clear the
// per-call accumulators themselves at its start.
static __device__ __align__(256) unsigned char g_noalloc_scratch[NoAllocLayout::total];

constexpr int kNoAllocMaxDevices = 64;

struct NoAllocDevice {
    bool ready = false;
    unsigned char* scratch = nullptr;   // device address of g_noalloc_scratch on this device
    int num_sms = 0;
    int smem_optin = 0;
};

NoAllocDevice g_noalloc_dev[kNoAllocMaxDevices];
std::mutex g_noalloc_mutex;

// Once per device, with that device current: look up the array's device
// address (in host code its name only stands in for it) and the SM limits.
lmloss_status noalloc_setup(int device, NoAllocDevice** out)
{
    std::lock_guard<std::mutex> lock(g_noalloc_mutex);
    NoAllocDevice& d = g_noalloc_dev[device];
    if (!d.ready) {
        void* ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || ptr == nullptr) {
            cudaGetLastError();
            return LMLOSS_ERR_CUDA;
        }
        if (cudaDeviceGetAttribute(&d.num_sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess ||
            cudaDeviceGetAttribute(&d.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, device) != cudaSuccess)
            return LMLOSS_ERR_CUDA;
        // the block counters must start at zero; the array is zero when the
        // module loads, and clearing it here states that rather than relying on it
        // (a synchronous memset of memory the library owns: no allocation)
        if (cudaMemset(ptr, 0, NoAllocLayout::total) != cudaSuccess) {
            cudaGetLastError();
            return LMLOSS_ERR_CUDA;
        }
        d.scratch = static_cast<unsigned char*>(ptr);
        d.ready = true;
    }
    *out = &d;
    return LMLOSS_OK;
}

}  // namespace

extern "C" lmloss_status lmloss_forward_backward_noalloc(const lmloss_args* a, cudaStream_t stream)
{
    lmloss_status st = check(a);
    if (st != LMLOSS_OK) return st;
    if (a->T > kNoAllocMaxT) return LMLOSS_ERR_INVALID_ARG;
    if (a->segment_ids && a->num_segments > kNoAllocMaxS) return LMLOSS_ERR_INVALID_ARG;
    int device = -1;
    if (cudaGetDevice(&device) != cudaSuccess) return LMLOSS_ERR_CUDA;
    if (device < 0 || device >= kNoAllocMaxDevices) return LMLOSS_ERR_UNSUPPORTED;
    NoAllocDevice* d = nullptr;
    if ((st = noalloc_setup(device, &d)) != LMLOSS_OK) return st;

    // A context on the stack whose workspace is the fixed array: the regular
    // call path then runs unchanged and allocates nothing.
    lmloss_ctx ctx;
    ctx.device = device;
    ctx.max_T = kNoAllocMaxT;
    ctx.max_S = static_cast<int32_t>(kNoAllocMaxS);
    ctx.num_sms = d->num_sms;
    ctx.smem_optin = d->smem_optin;
    unsigned char* b = d->scratch;
    using L = NoAllocLayout;
    ctx.ws.row_nll = reinterpret_cast<float*>(b + L::nll);
    ctx.ws.row_lse = reinterpret_cast<float*>(b + L::lse);
    ctx.ws.row_kl = reinterpret_cast<float*>(b + L::kl);
    ctx.ws.row_pol = reinterpret_cast<float*>(b + L::pol);
    ctx.ws.row_tu = reinterpret_cast<float*>(b + L::tu);
    ctx.ws.row_tt = reinterpret_cast<float*>(b + L::tt);
    ctx.ws.n_active = reinterpret_cast<int64_t*>(b + L::scal);
    ctx.ws.n_nonempty = reinterpret_cast<int64_t*>(b + L::scal + 8);
    ctx.ws.gspo_sum = reinterpret_cast<double*>(b + L::scal + 16);
    ctx.ws.s_seg = reinterpret_cast<double*>(b + L::scal + 24);
    ctx.ws.seg_n = reinterpret_cast<int*>(b + L::seg_n);
    ctx.ws.seg_dq = reinterpret_cast<unsigned long long*>(b + L::seg_dq);
    ctx.ws.seg_absq = reinterpret_cast<unsigned long long*>(b + L::seg_absq);
    ctx.ws.seg_nonfinite = reinterpret_cast<int*>(b + L::seg_nf);
    ctx.ws.seg_coef = reinterpret_cast<float*>(b + L::seg_coef);
    ctx.ws.row_counter = reinterpret_cast<int*>(b + L::counter);
    ctx.ws.cnt_part = reinterpret_cast<long long*>(b + L::cnt_part);
    ctx.ws.red_part = reinterpret_cast<double*>(b + L::red_part);
    ctx.ws.done = reinterpret_cast<unsigned*>(b + L::done);
    ctx.ws.err = reinterpret_cast<int*>(b + L::err);
    return lmloss_forward_backward(&ctx, a, stream);
}
