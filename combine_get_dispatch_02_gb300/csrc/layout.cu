// Dispatch layout kernel: counts, prefix sums and deterministic slots from
// topk_idx, in one launch of one thread-block cluster.
//
// What it computes is the layout DeepEP derives once per routing and reuses
// through the dispatch handle ("如何突破MoE通信瓶颈：DeepEP跨节点优化技术终极指南",
// section 技术解析, and section 核心API示例 for the handle): for every
// entry (g, k) of topk_idx its receive row, where the rows of expert e start
// at base[e] and hold its entries in ascending (g, k) order, plus the
// per-expert / per-(expert, source rank) / per-rank counts.
//
// Design (one GPU, R virtual ranks):
//   * One cluster of CL CTAs (16 when the device allows it) covers all tokens;
//     CTA c owns a contiguous token range, split again into one contiguous
//     range per warp, so (CTA, warp, lane) order is (g, k) order.
//   * Pass 1: each warp counts its entries per expert and per (expert,
//     source rank) in shared memory, aggregating equal keys with
//     __match_any_sync so one atomic per distinct key per 32 entries.
//   * The CTAs exchange their per-expert totals through distributed shared
//     memory after a hardware cluster barrier: every CTA gets the count of
//     each expert in lower-ranked CTAs and the grand totals (hence the bases),
//     with no global-memory atomics, no spin-waits and no second launch.
//   * Pass 2: each warp walks its entries again in order; an entry's row is
//     base + (entries of the expert before this warp) + (entries earlier in
//     this warp), the last term from __match_any_sync and a lane mask.
#include <cooperative_groups.h>

#include "ep_internal.cuh"

namespace cg = cooperative_groups;

namespace ep {

namespace {

constexpr size_t kMaxSmem = 227 * 1024;
constexpr int kMaxCluster = 16;

// Exclusive scan of one int per thread across the block; *total gets the sum.
// scan must hold NT/32 + 1 ints.  Ends with a barrier.
template <int NT>
__device__ int block_exclusive_scan(int v, int *scan, int *total) {
    constexpr int NW = NT / 32;
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    int x = v;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const int y = __shfl_up_sync(0xFFFFFFFFu, x, d);
        if (lane >= d) x += y;
    }
    if (lane == 31) scan[w] = x;
    __syncthreads();
    if (w == 0) {
        const int s = lane < NW ? scan[lane] : 0;
        int incl = s;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const int y = __shfl_up_sync(0xFFFFFFFFu, incl, d);
            if (lane >= d) incl += y;
        }
        if (lane < NW) scan[lane] = incl - s;
        if (lane == 31) scan[NW] = incl;
    }
    __syncthreads();
    const int excl = scan[w] + x - v;
    *total = scan[NW];
    __syncthreads();
    return excl;
}

// Sum over the cluster's CTAs of a shared-memory int at `off` (all peers'
// loads are issued before the first add), and the part from CTAs ranked
// below `crank`.
__device__ __forceinline__ int2 cluster_sum_below(cg::cluster_group &cluster, int32_t *base, int off,
                                                  int CL, int crank) {
    int v[kMaxCluster];
#pragma unroll
    for (int c = 0; c < kMaxCluster; ++c) v[c] = c < CL ? cluster.map_shared_rank(base, c)[off] : 0;
    int pre = 0, tot = 0;
#pragma unroll
    for (int c = 0; c < kMaxCluster; ++c) {
        pre += c < crank ? v[c] : 0;
        tot += v[c];
    }
    return make_int2(pre, tot);
}

template <int NT>
__global__ void __launch_bounds__(NT, 1) layout_kernel(const LayoutParams p) {
    // The dispatch kernel queued behind this one may start loading and
    // quantising token rows now; it waits for these results before it reads
    // any slot.
    pdl_launch_dependents();

    cg::cluster_group cluster = cg::this_cluster();
    const int CL = (int)cluster.num_blocks();
    const int crank = (int)cluster.block_rank();
    constexpr int NW = NT / 32;
    const int tid = threadIdx.x, w = tid >> 5, lane = tid & 31;
    const int E = p.E, R = p.R, K = p.K, T = p.T;
    const int N = (int)p.N;  // N*K < 2^31 (checked on the host)
    const int per = (E + CL - 1) / CL;

    extern __shared__ int32_t sm[];
    int32_t *hist_w = sm;                 // [NW][E] warp counts -> warp start positions
    int32_t *cta_hist = hist_w + NW * E;  // [E]     read by peer CTAs
    int32_t *hist_er = cta_hist + E;      // [E][R]  read by peer CTAs
    int32_t *tok_rank = hist_er + E * R;  // [R]     read by peer CTAs
    int32_t *epre = tok_rank + R;         // [E]     entries of e in lower CTAs
    int32_t *ebase = epre + E;            // [E]     totals, then first rows
    int32_t *scan = ebase + E;            // [NW+1]
    int32_t *pair = scan + NW + 1;        // [per][R]
    int16_t *stage = reinterpret_cast<int16_t *>(pair + per * R);  // [NW][tpw*K] expert ids

    const int zero_words = NW * E + E + E * R + R;
    for (int i = tid; i < zero_words; i += NT) sm[i] = 0;

    // contiguous token range per warp, warps of a CTA adjacent
    const int nwarps = CL * NW;
    const int tpw = (N + nwarps - 1) / nwarps;
    const int cta_t0 = min(N, crank * NW * tpw);
    const int cta_t1 = min(N, cta_t0 + NW * tpw);
    const int t0 = min(cta_t1, cta_t0 + w * tpw);
    const int t1 = min(cta_t1, t0 + tpw);
    const int i0 = t0 * K, i1 = t1 * K;
    // this warp's entry ids in shared memory for pass 2 (when they fit)
    int16_t *my_stage = p.staged ? stage + (size_t)w * tpw * K : nullptr;

    // membership rows of this CTA's tokens start at zero
    if (p.is_token_in_rank) {
        for (int b = cta_t0 * R + tid; b < cta_t1 * R; b += NT) p.is_token_in_rank[b] = 0;
    }
    __syncthreads();

    // ---------------- pass 1: counts (four loads in flight per lane)
    constexpr int kU = 4;
    for (int ib = i0; ib < i1; ib += 32 * kU) {
        int64_t ev[kU];
#pragma unroll
        for (int u = 0; u < kU; ++u) {
            const int i = ib + u * 32 + lane;
            ev[u] = i < i1 ? p.topk_idx[i] : -1;
        }
#pragma unroll
        for (int u = 0; u < kU; ++u) {
            const int i = ib + u * 32 + lane;
            const bool in = i < i1;
            const int64_t e = ev[u];
            const bool valid = in && e >= 0 && e < E;
            if (in && (e < -1 || e >= E)) atomicOr(p.status, kStatusBadExpert);
            if (in && my_stage) my_stage[i - i0] = valid ? (int16_t)e : (int16_t)-1;
            const int key = valid ? (int)e * R + (i / K) / T : -1;
            const uint32_t peers = __match_any_sync(0xFFFFFFFFu, key);
            if (valid && lane == __ffs(peers) - 1) {
                const int n = __popc(peers);
                atomicAdd(&hist_w[w * E + (int)e], n);
                atomicAdd(&hist_er[key], n);
            }
        }
    }
    if (p.tokens_per_rank || p.is_token_in_rank) {
        for (int g = t0 + lane; g < t1; g += 32) {
            const int64_t *row = p.topk_idx + (int64_t)g * K;
            for (int k = 0; k < K; ++k) {
                const int64_t e = row[k];
                if (e < 0 || e >= E) continue;
                const int d = (int)e / p.L;
                bool seen = false;
                for (int k2 = 0; k2 < k && !seen; ++k2) {
                    const int64_t e2 = row[k2];
                    seen = e2 >= 0 && e2 < E && (int)e2 / p.L == d;
                }
                if (seen) continue;
                atomicAdd(&tok_rank[d], 1);
                if (p.is_token_in_rank) p.is_token_in_rank[(int64_t)g * R + d] = 1;
            }
        }
    }
    __syncthreads();

    // per expert: exclusive prefix over this CTA's warps, and the CTA total
    for (int e = tid; e < E; e += NT) {
        int s = 0;
        for (int ww = 0; ww < NW; ++ww) {
            const int v = hist_w[ww * E + e];
            hist_w[ww * E + e] = s;
            s += v;
        }
        cta_hist[e] = s;
    }
    cluster.sync();  // every CTA's cta_hist / hist_er / tok_rank is final

    // per expert: entries in lower-ranked CTAs, and the total over the cluster
    for (int e = tid; e < E; e += NT) {
        const int2 pt = cluster_sum_below(cluster, cta_hist, e, CL, crank);
        epre[e] = pt.x;
        ebase[e] = pt.y;
    }
    // counts per (expert, source rank) for this CTA's slice of experts
    const int pe0 = min(E, crank * per), pe1 = min(E, pe0 + per);
    const int npairs = (pe1 - pe0) * R;
    for (int q = tid; q < npairs; q += NT) {
        const int j = pe0 * R + q;
        const int v = cluster_sum_below(cluster, hist_er, j, CL, 0).y;
        pair[q] = v;
        p.cnt_er[j] = v;
    }
    if (crank == 0 && p.tokens_per_rank) {
        for (int d = tid; d < R; d += NT) p.tokens_per_rank[d] = cluster_sum_below(cluster, tok_rank, d, CL, 0).y;
    }
    __syncthreads();

    // first row of each expert: e * cap (padded) or the exclusive prefix of
    // the totals (packed); CTA 0 publishes totals and bases
    {
        const int chunk = (E + NT - 1) / NT;
        const int e_lo = min(E, tid * chunk), e_hi = min(E, e_lo + chunk);
        int local = 0;
        for (int e = e_lo; e < e_hi; ++e) local += ebase[e];
        int total;
        int run = block_exclusive_scan<NT>(local, scan, &total);
        for (int e = e_lo; e < e_hi; ++e) {
            const int tot = ebase[e];
            const int b = p.layout == kLayoutPadded ? (int)(e * p.cap) : run;
            run += tot;
            if (crank == 0) {
                const int n = (int)min((int64_t)tot, p.cap);
                p.tokens_per_expert[e] = n;
                if (p.user_tokens_per_expert) p.user_tokens_per_expert[e] = n;
                p.base[e] = b;
            }
            ebase[e] = b;
        }
    }
    for (int e = pe0 + tid; e < pe1; e += NT) {
        int run = 0;
        for (int r = 0; r < R; ++r) {
            p.off_er[e * R + r] = run;
            run += pair[(e - pe0) * R + r];
        }
    }
    // start position of each warp within each expert
    for (int i = tid; i < NW * E; i += NT) hist_w[i] += epre[i % E];
    cluster.sync();  // peers are done reading this CTA's shared memory

    // ---------------- pass 2: rows, in (g, k) order
    const uint32_t lt = lanemask_lt();
    const int cap = (int)min(p.cap, (int64_t)0x7FFFFFFF);
    for (int ib = i0; ib < i1; ib += 32 * kU) {
        int ev[kU];
#pragma unroll
        for (int u = 0; u < kU; ++u) {
            const int i = ib + u * 32 + lane;
            if (i >= i1) {
                ev[u] = -1;
            } else if (my_stage) {
                ev[u] = my_stage[i - i0];
            } else {
                const int64_t e = p.topk_idx[i];
                ev[u] = (e >= 0 && e < E) ? (int)e : -1;
            }
        }
#pragma unroll
        for (int u = 0; u < kU; ++u) {
            const int i = ib + u * 32 + lane;
            const int e = ev[u];
            const bool valid = e >= 0;
            const uint32_t peers = __match_any_sync(0xFFFFFFFFu, e);
            int pos = 0;
            if (valid) pos = hist_w[w * E + e] + __popc(peers & lt);
            __syncwarp();
            if (valid && lane == __ffs(peers) - 1) hist_w[w * E + e] += __popc(peers);
            __syncwarp();
            if (i < i1) {
                int32_t s = -1;
                if (valid) {
                    if (pos < cap) {
                        s = ebase[e] + pos;
                        p.src_info[s] = i;
                    } else {
                        atomicOr(p.status, kStatusCapacity);
                    }
                }
                p.slot[i] = s;
            }
        }
    }
}

template <int NT>
cudaError_t launch_nt(LayoutParams p, int cl, cudaStream_t stream) {
    size_t smem = layout_smem_bytes(p.E, p.R, NT, cl);
    // stage the entries' expert ids in shared memory for the second pass
    // when they fit next to the histograms
    const int64_t nwarps = (int64_t)cl * (NT / 32);
    const int64_t tpw = (p.N + nwarps - 1) / nwarps;
    const size_t stage = (size_t)(NT / 32) * tpw * p.K * sizeof(int16_t);
    p.staged = (smem + stage <= kMaxSmem) ? 1 : 0;
    if (p.staged) smem += (stage + 15) / 16 * 16;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(cl, 1, 1);
    cfg.blockDim = dim3(NT, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = cl;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, layout_kernel<NT>, p);
}

template <int NT>
bool fits(int E, int R, int cl) {
    const size_t smem = layout_smem_bytes(E, R, NT, cl);
    if (smem > kMaxSmem) return false;
    auto k = layout_kernel<NT>;
    // the limit is set to the most any shape needs, so contexts of different
    // sizes can share the kernel
    if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kMaxSmem) != cudaSuccess ||
        cudaFuncSetAttribute(k, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(cl, 1, 1);
    cfg.blockDim = dim3(NT, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = cl;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, k, &cfg) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    return n >= 1;
}

}  // namespace

size_t layout_smem_bytes(int E, int R, int threads, int cluster_size) {
    const size_t NW = threads / 32;
    const size_t per = (E + cluster_size - 1) / cluster_size;
    const size_t words = NW * E + E + (size_t)E * R + R + E + E + (NW + 1) + per * R;
    return words * sizeof(int32_t);
}

bool layout_pick_shape(int E, int R, int *cluster_size, int *threads) {
    static const int cls[] = {16, 8, 4, 2, 1};
    for (int cl : cls) {
        if (fits<1024>(E, R, cl)) { *cluster_size = cl; *threads = 1024; return true; }
        if (fits<512>(E, R, cl)) { *cluster_size = cl; *threads = 512; return true; }
        if (fits<256>(E, R, cl)) { *cluster_size = cl; *threads = 256; return true; }
    }
    return false;
}

cudaError_t launch_layout(const LayoutParams &p, int cluster_size, int threads,
                          cudaStream_t stream) {
    switch (threads) {
        case 1024: return launch_nt<1024>(p, cluster_size, stream);
        case 512: return launch_nt<512>(p, cluster_size, stream);
        case 256: return launch_nt<256>(p, cluster_size, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace ep
