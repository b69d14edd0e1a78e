// The small kernels around the fused one: the count that gives the token
// scale and checks targets (K0), the merge of vocabulary-shard partials, the
// GSPO seam, the fixed-order loss reduction, and the bounded-wait self-test.
#pragma once

#include "kernels.cuh"

namespace lmloss {

// ======================================================================
// K0: count active rows, validate targets, clear the per-call accumulators.
// Block b counts a fixed chunk of rows; the last block to finish adds the
// block counts in block order.  Integer sums: deterministic.
// ======================================================================
__global__ void __launch_bounds__(256) count_kernel(const CallParams p)
{
    __shared__ long long part[8];
    __shared__ long long fin[kRedBlocks];
    __shared__ bool last;
    const int tid = threadIdx.x, nb = gridDim.x;
    const int64_t chunk = (p.T + nb - 1) / nb;
    const int64_t r0 = blockIdx.x * chunk, r1 = min(p.T, r0 + chunk);
    long long n = 0;
    for (int64_t r = r0 + tid; r < r1; r += blockDim.x) {
        int64_t t;
        if (row_active(p, r, t)) {
            ++n;
            if (t < 0 || t >= p.v_total) set_error(p.ws.err, kErrBadTarget);
        }
    }
    for (int i = blockIdx.x * blockDim.x + tid; i < p.num_segments; i += nb * blockDim.x) {
        p.ws.seg_n[i] = 0;
        p.ws.seg_dq[i] = 0ull;
        p.ws.seg_absq[i] = 0ull;
        p.ws.seg_nonfinite[3 * i] = 0;
        p.ws.seg_nonfinite[3 * i + 1] = 0;
        p.ws.seg_nonfinite[3 * i + 2] = 0;
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) n += __shfl_xor_sync(0xffffffffu, n, off);
    if ((tid & 31) == 0) part[tid >> 5] = n;
    __syncthreads();
    if (tid == 0) {
        long long v = 0;
        for (int k = 0; k < (blockDim.x >> 5); ++k) v += part[k];
        p.ws.cnt_part[blockIdx.x] = v;
        if (blockIdx.x == 0) {
            *p.ws.n_nonempty = 0;
            *p.ws.gspo_sum = 0.0;
            *p.ws.row_counter = 0;
        }
        __threadfence();
        last = atomicAdd(&p.ws.done[0], 1u) == static_cast<unsigned>(nb - 1);
    }
    __syncthreads();
    if (last) {
        // the last block: the block counts are loaded in parallel, then added
        __threadfence();
        if (tid < nb) fin[tid] = *reinterpret_cast<volatile long long*>(&p.ws.cnt_part[tid]);
        __syncthreads();
        if (tid == 0) {
            long long tot = 0;
            for (int k = 0; k < nb; ++k) tot += fin[k];
            *p.ws.n_active = tot;
            p.ws.done[0] = 0u;
        }
    }
}

// ======================================================================
// Vocabulary-split rows: the merge of the K shards' partials of each row
// (max M_k, sum S_k against it, target logit where the shard holds it) into
// the row's NLL and lse, as the record merge does across a cluster:
// M = max M_k, S = sum_k S_k e^(M_k - M) in shard order, then ce_scalars.
// torchtitan PR 5661, "Numerics (TP > 1 only)": each vocabulary shard drops
// the target from its own sum; only the statistics are combined.
// ======================================================================
struct ShardParts {
    const float* part[kMaxShards];   // [T, 4] each
    int K;
};

__global__ void __launch_bounds__(256) shard_merge_kernel(const CallParams p, const ShardParts sp)
{
    for (int64_t r = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; r < p.T;
         r += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        int64_t t;
        float nll = 0.f, lse = 0.f;
        if (row_active(p, r, t)) {
            float M = -INFINITY;
            for (int k = 0; k < sp.K; ++k) M = fmaxf(M, sp.part[k][4 * r]);
            float S = 0.f, zt = 0.f;
            int owners = 0;
            for (int k = 0; k < sp.K; ++k) {
                const float* q = sp.part[k] + 4 * r;
                if (q[1] != 0.f) S += q[1] * rescale(q[0], M);
                if (q[3] != 0.f) { zt = q[2]; ++owners; }
            }
            if (owners != 1 || t < 0 || t >= p.v_total) {
                // target outside [0, V) (flagged by the count) or held by no shard
                if (owners != 1) set_error(p.ws.err, kErrBadTarget);
                nll = lse = __int_as_float(0x7fc00000);
            } else {
                float lnS, sp_neg, pt, pnt;
                ce_scalars(M, S, zt, nll, lse, lnS, sp_neg, pt, pnt);
            }
        }
        p.ws.row_nll[r] = nll;
        p.ws.row_lse[r] = lse;
        p.ws.row_kl[r] = 0.f;
        p.ws.row_pol[r] = 0.f;
        if (p.logp_out) p.logp_out[r] = -nll;
        if (p.lse_out) p.lse_out[r] = lse;
    }
}

// ======================================================================
// GSPO seam, part 1: per-token index-add of counts and log-ratios into the
// segment accumulators.  Fixed-point integer sums make the result independent
// of the order in which tokens arrive.
// Fast-LLM PR 552 "Fuse GSPO into the monolithic compiled loss (#507)",
// "Why it needed special handling": index_add over num_segments, then clipping.
// ======================================================================
__global__ void seam_accum_kernel(const CallParams p)
{
    for (int64_t r = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; r < p.T;
         r += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        int64_t t;
        if (!row_active(p, r, t)) continue;
        const int g = p.seg_ids[r];
        if (g < 0) continue;
        if (g >= p.num_segments) { set_error(p.ws.err, kErrBadSegment); continue; }
        atomicAdd(&p.ws.seg_n[g], 1);
        const double x = -static_cast<double>(p.ws.row_nll[r]) - static_cast<double>(p.old_logp[r]);
        if (isnan(x)) { atomicAdd(&p.ws.seg_nonfinite[3 * g + 2], 1); continue; }
        if (isinf(x)) { atomicAdd(&p.ws.seg_nonfinite[3 * g + (x > 0 ? 0 : 1)], 1); continue; }
        if (fabs(x) >= 1073741824.0) { set_error(p.ws.err, kErrRange); continue; }
        const long long q = __double2ll_rn(x * 4294967296.0);
        atomicAdd(&p.ws.seg_dq[g], static_cast<unsigned long long>(q));
        atomicAdd(&p.ws.seg_absq[g], static_cast<unsigned long long>(fabs(x) * 256.0));
    }
}

// ======================================================================
// GSPO seam, part 2 (one CTA): ratio, clipping, loss and gradient coefficient
// per segment; the GSPO scale; a fixed-order sum of the segment losses.
// ======================================================================
__global__ void __launch_bounds__(1024) seam_finish_kernel(const CallParams p)
{
    __shared__ double dpart[32];
    __shared__ long long ipart[32];
    __shared__ double s_seg_sh;
    const int S = p.num_segments;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nw = blockDim.x >> 5;

    long long ne = 0;
    for (int i = tid; i < S; i += blockDim.x) ne += (p.ws.seg_n[i] > 0) ? 1 : 0;
    for (int off = 16; off > 0; off >>= 1) ne += __shfl_xor_sync(0xffffffffu, ne, off);
    if (lane == 0) ipart[warp] = ne;
    __syncthreads();
    if (tid == 0) {
        long long tot = 0;
        for (int k = 0; k < nw; ++k) tot += ipart[k];
        *p.ws.n_nonempty = tot;
        *p.ws.row_counter = 0;   // the gradient pass hands out rows afresh
        s_seg_sh = (p.reduction == 1) ? (tot > 0 ? 1.0 / static_cast<double>(tot) : 0.0) : p.inv_denominator;
        *p.ws.s_seg = s_seg_sh;
    }
    __syncthreads();
    const double s_seg = s_seg_sh;
    const double lo = 1.0 - static_cast<double>(p.eps_lo), hi = 1.0 + static_cast<double>(p.eps_hi);

    double lsum = 0.0;
    for (int i = tid; i < S; i += blockDim.x) {
        const int n = p.ws.seg_n[i];
        float ratio = 0.f, lossf = 0.f, coef = 0.f;
        uint8_t flag = 0;
        if (n > 0) {
            const int* nf = &p.ws.seg_nonfinite[3 * i];
            double D;
            if (nf[2] > 0 || (nf[0] > 0 && nf[1] > 0)) D = __longlong_as_double(0x7ff8000000000000LL);
            else if (nf[0] > 0) D = __longlong_as_double(0x7ff0000000000000LL);
            else if (nf[1] > 0) D = -__longlong_as_double(0x7ff0000000000000LL);
            else {
                if (p.ws.seg_absq[i] >= (1ull << 38)) set_error(p.ws.err, kErrRange);
                D = static_cast<double>(static_cast<long long>(p.ws.seg_dq[i])) * (1.0 / 4294967296.0);
            }
            const double A = static_cast<double>(p.adv[i]);
            const double s = exp(D / n);
            const double c = fmin(fmax(s, lo), hi);
            const double L = -fmin(s * A, c * A);
            flag = (s * A <= c * A) ? 1 : 0;
            ratio = static_cast<float>(s);
            lossf = static_cast<float>(L);
            coef = flag ? static_cast<float>(s_seg * A * s / n) : 0.f;
            lsum += L;
        }
        p.ws.seg_coef[i] = coef;
        if (p.seg_count_out) p.seg_count_out[i] = n;
        if (p.seg_ratio_out) p.seg_ratio_out[i] = ratio;
        if (p.seg_flag_out) p.seg_flag_out[i] = flag;
        if (p.seg_loss_out) p.seg_loss_out[i] = lossf;
    }
    for (int off = 16; off > 0; off >>= 1) lsum += __shfl_xor_sync(0xffffffffu, lsum, off);
    if (lane == 0) dpart[warp] = lsum;
    __syncthreads();
    if (tid == 0) {
        double tot = 0.0;
        for (int k = 0; k < nw; ++k) tot += dpart[k];
        *p.ws.gspo_sum = tot;
    }
}

// ======================================================================
// K4: deterministic loss reduction.  Block b sums a fixed chunk of rows in a
// fixed order (fp64); the last block to finish adds the block partials in
// block order and scales them.
// xtuner PR 1963 "[FSDP][Loss] Switch gradient reduction to SUM": each term
// is its sum over tokens times the reduction scale; the z term carries alpha
// (z-loss diff: loss * z_loss_alpha / batch_size).
// ======================================================================
__global__ void __launch_bounds__(256) reduce_kernel(const CallParams p)
{
    __shared__ double part[4][8];
    __shared__ long long npart[8];
    __shared__ double fin[4][kRedBlocks];
    __shared__ long long nfin[kRedBlocks];   // one per warp of the last block's tree
    __shared__ bool last;
    // may be launched while the staged-row kernel before it still runs: its
    // per-row results must be complete and visible before any is read
    grid_dep_wait();
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nw = blockDim.x >> 5, nb = gridDim.x;
    const int64_t chunk = (p.T + nb - 1) / nb;
    const int64_t r0 = blockIdx.x * chunk, r1 = min(p.T, r0 + chunk);
    double a = 0.0, b = 0.0, c = 0.0, d = 0.0;
    long long n = 0;   // active rows, counted here too: calls under SUM run no count kernel
    for (int64_t r = r0 + tid; r < r1; r += blockDim.x) {
        const double lse = p.ws.row_lse[r];
        a += p.ws.row_nll[r];
        b += lse * lse;
        c += p.ws.row_kl[r];
        if (p.tok_adv) d += p.ws.row_pol[r];
        int64_t t;
        n += row_active(p, r, t) ? 1 : 0;
    }
    for (int off = 16; off > 0; off >>= 1) {
        a += __shfl_xor_sync(0xffffffffu, a, off);
        b += __shfl_xor_sync(0xffffffffu, b, off);
        c += __shfl_xor_sync(0xffffffffu, c, off);
        d += __shfl_xor_sync(0xffffffffu, d, off);
        n += __shfl_xor_sync(0xffffffffu, n, off);
    }
    if (lane == 0) { part[0][warp] = a; part[1][warp] = b; part[2][warp] = c; part[3][warp] = d; npart[warp] = n; }
    __syncthreads();
    // the block's warps, then the blocks, are added by fixed-shape shuffle trees:
    // the same order on every call, and log2 depth instead of a serial chain
    // of double additions (a slow pipe on this GPU)
    if (warp == 0) {
        a = (lane < nw) ? part[0][lane] : 0.0;
        b = (lane < nw) ? part[1][lane] : 0.0;
        c = (lane < nw) ? part[2][lane] : 0.0;
        d = (lane < nw) ? part[3][lane] : 0.0;
        n = (lane < nw) ? npart[lane] : 0;
        for (int off = 16; off > 0; off >>= 1) {
            a += __shfl_xor_sync(0xffffffffu, a, off);
            b += __shfl_xor_sync(0xffffffffu, b, off);
            c += __shfl_xor_sync(0xffffffffu, c, off);
            d += __shfl_xor_sync(0xffffffffu, d, off);
            n += __shfl_xor_sync(0xffffffffu, n, off);
        }
        if (lane == 0) {
            p.ws.red_part[4 * blockIdx.x] = a;
            p.ws.red_part[4 * blockIdx.x + 1] = b;
            p.ws.red_part[4 * blockIdx.x + 2] = c;
            p.ws.red_part[4 * blockIdx.x + 3] = d;
            p.ws.cnt_part[blockIdx.x] = n;
            __threadfence();
            last = atomicAdd(&p.ws.done[1], 1u) == static_cast<unsigned>(nb - 1);
        }
    }
    __syncthreads();
    if (!last) return;
    // the last block: the block partials are loaded in parallel and added by
    // the same fixed-shape shuffle tree (counts with them), then one thread adds
    // the two warps' sums: the same order on every call
    __threadfence();
    if (tid < kRedBlocks) {
        double v0 = 0.0, v1 = 0.0, v2 = 0.0, v3 = 0.0;
        long long c = 0;
        if (tid < nb) {
            const volatile double* rp = p.ws.red_part + 4 * tid;
            v0 = rp[0]; v1 = rp[1]; v2 = rp[2]; v3 = rp[3];
            c = *reinterpret_cast<volatile long long*>(&p.ws.cnt_part[tid]);
        }
        for (int off = 16; off > 0; off >>= 1) {
            v0 += __shfl_xor_sync(0xffffffffu, v0, off);
            v1 += __shfl_xor_sync(0xffffffffu, v1, off);
            v2 += __shfl_xor_sync(0xffffffffu, v2, off);
            v3 += __shfl_xor_sync(0xffffffffu, v3, off);
            c += __shfl_xor_sync(0xffffffffu, c, off);
        }
        if (lane == 0) {
            fin[0][warp] = v0; fin[1][warp] = v1; fin[2][warp] = v2; fin[3][warp] = v3;
            nfin[warp] = c;
        }
    }
    __syncthreads();
    if (tid == 0) {
        double sa = 0.0, sb = 0.0, sc = 0.0, sd = 0.0;
        long long n = 0;
        for (int k = 0; k < kRedBlocks / 32; ++k) {
            sa += fin[0][k]; sb += fin[1][k]; sc += fin[2][k]; sd += fin[3][k];
            n += nfin[k];
        }
        p.ws.done[1] = 0u;
        const double s = (p.reduction == 1) ? (n > 0 ? 1.0 / static_cast<double>(n) : 0.0) : p.inv_denominator;
        const double ce = s * sa;
        const double z = s * static_cast<double>(p.alpha) * sb;
        const double kl = s * sc;
        double gspo = 0.0;                       // the policy term: GSPO or GRPO
        if (p.seg_ids) gspo = *p.ws.s_seg * *p.ws.gspo_sum;
        else if (p.tok_adv) gspo = s * sd;
        const double total = static_cast<double>(p.w_ce) * ce + z + static_cast<double>(p.w_kl) * kl + gspo;
        p.loss_out[0] = static_cast<float>(total);
        p.loss_out[1] = static_cast<float>(ce);
        p.loss_out[2] = static_cast<float>(z);
        p.loss_out[3] = static_cast<float>(kl);
        p.loss_out[4] = static_cast<float>(gspo);
        if (p.count_out) {
            p.count_out[0] = n;
            p.count_out[1] = p.seg_ids ? *p.ws.n_nonempty : 0;
        }
    }
}

// ======================================================================
// Self-test of the bounded wait used by every kernel above: one thread waits
// on an mbarrier that nothing ever arrives at, with the given limit, and
// records whether the wait gave up.  Nothing is copied, so nothing is left in
// flight when it returns.
// ======================================================================
__global__ void wait_selftest_kernel(long long limit_cycles, int* status)
{
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(smem_addr(&bar), 1);
        fence_mbar_init();
        const bool done = mbar_wait_bounded(smem_addr(&bar), 0u, limit_cycles);
        *status = done ? 0 : kErrTimeout;
    }
}

}  // namespace lmloss
