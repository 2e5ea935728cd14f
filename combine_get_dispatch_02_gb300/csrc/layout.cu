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
//   * Equal keys inside a warp are found with one ballot per key bit (a
//     deterministic multi-split: lanes whose bits all agree hold the same
//     key), which is much cheaper than match.any on this GPU.
//   * Pass 1: each warp counts its entries per expert in shared memory.  Each
//     CTA then stores its per-expert totals into every peer's shared memory
//     (distributed shared memory) and, after one hardware cluster barrier,
//     every CTA holds all totals locally: its prefix, the grand totals and the
//     bases follow without global atomics, spin-waits or a second launch.
//   * Pass 1 also records each entry's position among its warp's entries of
//     the same expert (in a shared-memory copy of the warp's entries when it
//     fits), so pass 2 needs no cross-lane work: an entry's row is base +
//     (entries of the expert in lower CTAs) + (in lower warps) + (its
//     position in the warp).  Without the copy pass 2 re-derives the
//     positions from topk_idx.
//   * Per-(expert, source rank) ranges (cnt_er / off_er) are optional: pass 1
//     also counts per (expert, source rank) in shared memory, each CTA adds
//     its counts to the zeroed global cnt_er after the cluster barrier, and
//     after a second barrier the owner CTAs turn them into offsets.
#include <cooperative_groups.h>

#include "ep_internal.cuh"

namespace cg = cooperative_groups;

namespace ep {

namespace {

constexpr size_t kMaxSmem = 227 * 1024;
constexpr int kU = 4;  // 32-entry rounds per warp in flight

// Lanes of the warp whose key equals this lane's (all lanes take part; keys
// are non-negative and below 2^nbits).
__device__ __forceinline__ uint32_t warp_match(int key, int nbits) {
    uint32_t m = 0xFFFFFFFFu;
    for (int b = 0; b < nbits; ++b) {
        const bool bit = (key >> b) & 1;
        const uint32_t v = __ballot_sync(0xFFFFFFFFu, bit);
        m &= bit ? v : ~v;
    }
    return m;
}

__device__ __forceinline__ int bits_for(int n) {  // smallest b with n <= 2^b
    return 32 - __clz(max(n - 1, 1));
}

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

// Raw topk_idx entry i, or -1 past the end (no branch on the loaded value, so
// several of these stay in flight).
__device__ __forceinline__ int64_t load_raw(const int64_t *idx, int i, int i1) {
    return i < i1 ? __ldg(idx + i) : -1;
}

// Key of entry i with raw id e: its expert, or in rank mode the rank that
// owns the expert when no earlier k of the same token goes to that rank; -1
// for none.  Ids outside [-1, num_experts) are flagged and skipped.  Called
// by all 32 lanes of a warp on 32 consecutive entries that start at a token
// boundary (rounds of 32 entries from a token-aligned start): when K divides
// 32 the earlier entries of a lane's token are the K - 1 lanes before it, so
// rank mode compares with them by shuffles instead of re-reading topk_idx.
__device__ __forceinline__ int to_key(const LayoutParams &p, int64_t e, int i) {
    const bool valid = e >= 0 && e < p.num_experts;
    if (!valid && e != -1) atomicOr(p.status, kStatusBadExpert);
    if (!p.rank_mode) return valid ? (int)e : -1;
    const int d = valid ? (int)e / p.L : -1;
    if ((32 % p.K) == 0) {  // warp-uniform
        const int kk = i % p.K;  // this entry's k
        bool first = d >= 0;
        for (int s = 1; s < p.K; ++s) {
            const int dp = __shfl_up_sync(0xFFFFFFFFu, d, s);
            if (s <= kk && dp == d) first = false;
        }
        return first ? d : -1;
    }
    if (d < 0) return -1;
    for (int j = (i / p.K) * p.K; j < i; ++j) {
        const int64_t e2 = __ldg(p.topk_idx + j);
        if (e2 >= 0 && e2 < p.num_experts && (int)e2 / p.L == d) return -1;
    }
    return d;
}

template <int NT>
__global__ void __launch_bounds__(NT, 1) layout_kernel(const LayoutParams p) {
    // The dispatch kernel queued behind this one may start loading and
    // quantising token rows now; it waits for these results before it reads
    // any slot.
    pdl_launch_dependents();
    // peers may write into this CTA's shared memory only once every CTA of
    // the cluster is running: arrive now, wait just before the first push
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");

    cg::cluster_group cluster = cg::this_cluster();
    const int CL = (int)cluster.num_blocks();
    const int crank = (int)cluster.block_rank();
    constexpr int NW = NT / 32;
    const int tid = threadIdx.x, w = tid >> 5, lane = tid & 31;
    const int E = p.E, R = p.R, K = p.K, T = p.T;
    const int N = (int)p.N;  // N*K < 2^31 (checked on the host)
    const int ebits = bits_for(E + 1);  // keys 0..E-1 and E for "none"

    extern __shared__ int32_t sm[];
    int32_t *hist_w = sm;                   // [NW][E] warp counts -> warp start positions
    int32_t *tok_rank = hist_w + NW * E;    // [R]     this CTA's tokens per rank
    int32_t *recv_hist = tok_rank + R;      // [CL][E] per-expert totals of every CTA (pushed)
    int32_t *recv_tok = recv_hist + CL * E; // [CL][R] tokens per rank of every CTA (pushed to CTA 0)
    int32_t *epre = recv_tok + CL * R;      // [E]     entries of e in lower CTAs
    int32_t *ebase = epre + E;              // [E]     first row of e
    int32_t *scan = ebase + E;              // [NW+1]
    const int span = p.er_span;             // source ranks one CTA's tokens can cover (0: no ranges)
    int32_t *hist_er = scan + NW + 1;       // [E][span] entries per (expert, rank - first rank)
    int32_t *stage = hist_er + E * span;    // [NW][tpw*K] (position in warp << 11) | (expert + 1)

    // contiguous token range per warp, warps of a CTA adjacent
    const int nwarps = CL * NW;
    const int tpw = (N + nwarps - 1) / nwarps;
    const int cta_t0 = min(N, crank * NW * tpw);
    const int cta_t1 = min(N, cta_t0 + NW * tpw);
    const int t0 = min(cta_t1, cta_t0 + w * tpw);
    const int t1 = min(cta_t1, t0 + tpw);
    const int i0 = t0 * K, i1 = t1 * K;
    // (position, expert) of each entry between the passes: in shared memory
    // when it fits, else in the entry's own slot cell (the same thread writes
    // and later overwrites it)
    int32_t *my_stage = p.staged ? stage + (size_t)w * tpw * K : p.slot + i0;
    const bool want_er = p.cnt_er != nullptr;
    const int r0 = T > 0 ? cta_t0 / T : 0;  // first source rank of this CTA

    // first batch of entries in flight while shared memory is cleared
    int64_t raw[kU];
#pragma unroll
    for (int u = 0; u < kU; ++u) raw[u] = load_raw(p.topk_idx, i0 + u * 32 + lane, i1);

    for (int i = tid; i < NW * E + R; i += NT) sm[i] = 0;
    for (int i = tid; i < E * span; i += NT) hist_er[i] = 0;
    if (p.is_token_in_rank) {
        for (int b = cta_t0 * R + tid; b < cta_t1 * R; b += NT) p.is_token_in_rank[b] = 0;
    }
    if (p.cnt_er != nullptr) {  // owners clear their slice of the global (e, r) counts
        const int per = (E + CL - 1) / CL;
        const int j0 = min(E, crank * per) * R, j1 = min(E, crank * per + per) * R;
        for (int j = j0 + tid; j < j1; j += NT) p.cnt_er[j] = 0;
    }
    __syncthreads();

    // ---------------- pass 1: per-warp counts per expert
    const int erbits = bits_for(E * span + 1);
    for (int ib = i0; ib < i1; ib += 32 * kU) {
        if (ib != i0) {
#pragma unroll
            for (int u = 0; u < kU; ++u) raw[u] = load_raw(p.topk_idx, ib + u * 32 + lane, i1);
        }
#pragma unroll
        for (int u = 0; u < kU; ++u) {
            if (ib + u * 32 >= i1) break;  // warp-uniform
            const int i = ib + u * 32 + lane;
            const int e = to_key(p, raw[u], i);
            const uint32_t peers = warp_match(e < 0 ? E : e, ebits);
            // position of this entry among the warp's entries of expert e
            int local = 0;
            if (e >= 0) local = hist_w[w * E + e] + __popc(peers & lanemask_lt());
            __syncwarp();
            if (e >= 0 && lane == __ffs(peers) - 1) hist_w[w * E + e] += __popc(peers);
            __syncwarp();
            if (i < i1) my_stage[i - i0] = (local << 11) | (e + 1);
            if (want_er) {  // entries per (expert, source rank), one atomic per key per round
                const int key = e >= 0 ? e * span + (i / K) / T - r0 : E * span;
                const uint32_t pk = warp_match(key, erbits);
                if (e >= 0 && lane == __ffs(pk) - 1) atomicAdd(&hist_er[key], __popc(pk));
            }
        }
    }
    if (p.tokens_per_rank || p.is_token_in_rank) {
        for (int g = t0 + lane; g < t1; g += 32) {
            const int64_t *row = p.topk_idx + (int64_t)g * K;
            for (int k = 0; k < K; ++k) {
                const int64_t e = row[k];
                if (e < 0 || e >= p.num_experts) continue;
                const int d = (int)e / p.L;
                bool seen = false;
                for (int k2 = 0; k2 < k && !seen; ++k2) {
                    const int64_t e2 = row[k2];
                    seen = e2 >= 0 && e2 < p.num_experts && (int)e2 / p.L == d;
                }
                if (seen) continue;
                atomicAdd(&tok_rank[d], 1);
                if (p.is_token_in_rank) p.is_token_in_rank[(int64_t)g * R + d] = 1;
            }
        }
    }
    __syncthreads();

    // per expert: exclusive prefix over this CTA's warps; the CTA total goes
    // to every CTA of the cluster (slot crank of their recv_hist)
    asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
    for (int e = tid; e < E; e += NT) {
        int s = 0;
        for (int ww = 0; ww < NW; ++ww) {
            const int v = hist_w[ww * E + e];
            hist_w[ww * E + e] = s;
            s += v;
        }
        for (int c = 0; c < CL; ++c) cluster.map_shared_rank(recv_hist, c)[crank * E + e] = s;
    }
    if (p.tokens_per_rank) {
        int32_t *dst = cluster.map_shared_rank(recv_tok, 0);
        for (int d = tid; d < R; d += NT) dst[crank * R + d] = tok_rank[d];
    }
    cluster.sync();  // every CTA's totals are in every CTA's shared memory

    // per expert: entries in lower-ranked CTAs, and the total over the cluster
    for (int e = tid; e < E; e += NT) {
        int pre = 0, tot = 0;
        for (int c = 0; c < CL; ++c) {
            const int v = recv_hist[c * E + e];
            pre += c < crank ? v : 0;
            tot += v;
        }
        epre[e] = pre;
        ebase[e] = tot;
    }
    if (crank == 0 && p.tokens_per_rank) {
        for (int d = tid; d < R; d += NT) {
            int v = 0;
            for (int c = 0; c < CL; ++c) v += recv_tok[c * R + d];
            p.tokens_per_rank[d] = v;
        }
    }
    if (want_er) {  // the owners cleared cnt_er before the cluster barrier
        for (int j = tid; j < E * span; j += NT) {
            const int v = hist_er[j];
            if (v != 0) atomicAdd(&p.cnt_er[(j / span) * R + r0 + j % span], v);
        }
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
    __syncthreads();

    // ---------------- pass 2: rows, in (g, k) order
    // every entry's position inside its warp is known: rows follow directly
    const int cap = (int)min(p.cap, (int64_t)0x7FFFFFFF);
    for (int i = i0 + lane; i < i1; i += 32) {
        const int v = my_stage[i - i0];
        const int e = (v & 2047) - 1;
        int32_t s = -1;
        if (e >= 0) {
            const int pos = epre[e] + hist_w[w * E + e] + (v >> 11);
            if (pos < cap) {
                s = ebase[e] + pos;
                p.src_info[s] = i;
                if (p.recv_topk_idx != nullptr) {  // rank mode: the token's experts on rank e
                    const int g0 = (i / K) * K;
                    for (int k2 = 0; k2 < K; ++k2) {
                        const int64_t e2 = __ldg(p.topk_idx + g0 + k2);
                        const bool on = e2 >= 0 && e2 < p.num_experts && (int)e2 / p.L == e;
                        p.recv_topk_idx[(int64_t)s * K + k2] = on ? (int)e2 - e * p.L : -1;
                        if (p.recv_topk_weights != nullptr)
                            p.recv_topk_weights[(int64_t)s * K + k2] =
                                on ? (p.topk_weights != nullptr ? __ldg(p.topk_weights + g0 + k2) : 1.0f) : 0.0f;
                    }
                }
            } else {
                atomicOr(p.status, kStatusCapacity);
            }
        }
        p.slot[i] = s;
    }

    if (want_er) {
        cluster.sync();  // every CTA's (e, r) counts have landed in global memory
        // owners: off_er[e][r] = exclusive prefix over r, one warp per expert
        const int per = (E + CL - 1) / CL;
        const int pe0 = min(E, crank * per), pe1 = min(E, pe0 + per);
        for (int e = pe0 + w; e < pe1; e += NW) {
            int run = 0;
            for (int r0 = 0; r0 < R; r0 += 32) {
                const int r = r0 + lane;
                const int v = r < R ? __ldcg(&p.cnt_er[e * R + r]) : 0;
                int x = v;
#pragma unroll
                for (int d = 1; d < 32; d <<= 1) {
                    const int y = __shfl_up_sync(0xFFFFFFFFu, x, d);
                    if (lane >= d) x += y;
                }
                if (r < R) p.off_er[e * R + r] = run + x - v;
                run += __shfl_sync(0xFFFFFFFFu, x, 31);
            }
        }
    }
}

size_t smem_words(int E, int R, int NT, int CL) {
    const size_t NW = NT / 32;
    return NW * E + R + (size_t)CL * E + (size_t)CL * R + 2 * (size_t)E + NW + 1;
}

// Source ranks the token range of one CTA can touch (0 when no per-rank
// ranges are wanted).
int er_span_of(const LayoutParams &p, int NT, int CL) {
    if (p.cnt_er == nullptr) return 0;
    if (p.T <= 0) return 1;
    const int64_t nwarps = (int64_t)CL * (NT / 32);
    const int64_t tpw = (p.N + nwarps - 1) / nwarps;
    const int64_t span = (tpw * (NT / 32) + p.T - 1) / p.T + 1;
    return (int)(span < p.R ? span : p.R);
}

// stage bytes for the per-warp copies of the entries' expert ids
size_t stage_bytes(int64_t N, int K, int NT, int CL) {
    const int64_t nwarps = (int64_t)CL * (NT / 32);
    const int64_t tpw = (N + nwarps - 1) / nwarps;
    return (size_t)(NT / 32) * tpw * K * sizeof(int32_t);
}

template <int NT>
cudaError_t launch_nt(LayoutParams p, int cl, cudaStream_t stream) {
    {   // an entry's position in its warp is packed into 20 bits between the passes
        const int64_t nwarps = (int64_t)cl * (NT / 32);
        if ((p.N + nwarps - 1) / nwarps * p.K >= (int64_t(1) << 20)) return cudaErrorInvalidConfiguration;
    }
    p.er_span = er_span_of(p, NT, cl);
    size_t smem = (smem_words(p.E, p.R, NT, cl) + (size_t)p.E * p.er_span) * sizeof(int32_t);
    if (smem > kMaxSmem) return cudaErrorInvalidConfiguration;
    const size_t stage = stage_bytes(p.N, p.K, NT, cl);
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
    const size_t smem = smem_words(E, R, NT, cl) * sizeof(int32_t);
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

// ---------------------------------------------------------------- grid form
// The same layout for many entries from ONE cooperative kernel over the whole
// GPU (the single cluster above uses 16 SMs), C CTAs, all resident at once
// (cooperative launch), with two grid barriers:
//   count    pass 1 over the CTA's token range, as in the cluster kernel:
//            each entry's (position among its warp's entries of its key,
//            key) is staged in its slot cell, the warp prefixes stay in
//            shared memory, the CTA's key totals go to cta_hist[c][key]
//   barrier
//   scan     CTA c owns keys [c*E/C, (c+1)*E/C): per owned key one block scan
//            over the C CTA totals turns cta_hist[.][key] into entries of the
//            key in lower CTAs; totals, counts, padded bases, per-(expert,
//            rank) offsets
//   barrier
//   write    packed bases (a block scan of the totals, in every CTA), then
//            slot = base + prefix + position, src_info, rank-mode rows
// The barriers are one counter (zero between launches: the last CTA to leave
// puts it back); each wait is bounded (about one second): on expiry the
// kernel sets kStatusTimeout, still counts the arrivals it owes and leaves.
// The counts the layout accumulates with atomics are zeroed in the kernel
// before the first barrier and accumulated after it, so no host-side copy
// precedes the launch.  The dispatch queued behind (programmatic dependent launch) may
// start casting rows at once.
// threads per CTA of the grid form: 1024 from kGridBigEntries entries on (more
// warps per CTA shorten the count and write phases), 512 below (cheaper
// block scans and barriers when each CTA holds few entries)
constexpr int kGridBigEntries = 262144;
constexpr uint64_t kGridWaitNs = 1000000000ull;

__device__ __forceinline__ uint64_t grid_now_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
__device__ __forceinline__ uint32_t ld_acquire_gpu(const uint32_t *p) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void red_add_release_gpu(uint32_t *p, uint32_t v) {
    asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Arrive at the grid barrier and wait (bounded) until `target` CTAs have
// arrived.  Every CTA of the grid is resident (cooperative launch), so the
// wait ends unless something is broken.  False when it gave up.
__device__ bool grid_barrier(uint32_t *bar, uint32_t target, int *flag) {
    __syncthreads();
    if (threadIdx.x == 0) {
        // the arrival releases this CTA's writes (ordered before it by the
        // CTA barrier above); the polling load acquires the other CTAs'
        red_add_release_gpu(bar, 1u);
        bool ok = true;
        const uint64_t t0 = grid_now_ns();
        while (ld_acquire_gpu(bar) < target) {
            if (grid_now_ns() - t0 > kGridWaitNs) {
                ok = false;
                break;
            }
        }
        *flag = ok ? 1 : 0;
    }
    __syncthreads();
    return *flag != 0;
}

// Leaving the grid's barriers (thread 0 of a CTA): one more count per CTA,
// and the last of the 3C counts (C arrivals at each of the two barriers, C
// departures) puts the counter back to zero for the next launch.  A CTA
// that gave up waiting still adds every count it owes (`owed` arrivals it
// skipped, then its departure), so the counter always ends at zero.
__device__ void grid_depart(uint32_t *bar, uint32_t C, uint32_t owed) {
    const uint32_t old = atomicAdd(bar, owed + 1u);
    if (old + owed + 1u == 3u * C) atomicExch(bar, 0u);
}

template <int NT>
__global__ void __launch_bounds__(NT, 1) layout_grid_kernel(const LayoutParams p) {
    // the dispatch kernel queued behind this one may start loading and
    // casting token rows now; it waits for these results before it reads a slot
    pdl_launch_dependents();
    constexpr int NW = NT / 32;
    const int tid = threadIdx.x, w = tid >> 5, lane = tid & 31;
    const int E = p.E, R = p.R, K = p.K, T = p.T;
    const int N = (int)p.N;
    const int c = blockIdx.x, C = gridDim.x;
    const int ebits = bits_for(E + 1);
    extern __shared__ int32_t sm[];
    int32_t *hist_w = sm;                 // [NW][E] warp counts -> warp start positions in the CTA
    int32_t *tok_rank = hist_w + NW * E;  // [R]
    const int span = p.er_span;
    int32_t *hist_er = tok_rank + R;      // [E][span] (at least [E]: the bases in the write phase)
    int32_t *pre = hist_er + max(E * span, E);  // [E] entries of each key in lower CTAs
    int32_t *scan = pre + E;              // [NW + 1]
    __shared__ int bar_ok;
    const int cta_t0 = min(N, c * p.grid_tpc), cta_t1 = min(N, cta_t0 + p.grid_tpc);
    const int tpw = (p.grid_tpc + NW - 1) / NW;
    const int t0 = min(cta_t1, cta_t0 + w * tpw), t1 = min(cta_t1, t0 + tpw);
    const int i0 = t0 * K, i1 = t1 * K;
    int32_t *stage = p.slot;  // (position in warp, key) of each entry until the write phase
    const bool want_er = p.cnt_er != nullptr;
    const int r0 = T > 0 ? cta_t0 / T : 0;

    // ---------------- count
    int64_t raw[kU];
#pragma unroll
    for (int u = 0; u < kU; ++u) raw[u] = load_raw(p.topk_idx, i0 + u * 32 + lane, i1);
    for (int i = tid; i < NW * E + R; i += NT) sm[i] = 0;
    for (int i = tid; i < E * span; i += NT) hist_er[i] = 0;
    if (p.is_token_in_rank) {
        for (int b = cta_t0 * R + tid; b < cta_t1 * R; b += NT) p.is_token_in_rank[b] = 0;
    }
    __syncthreads();
    const int erbits = bits_for(E * span + 1);
    for (int ib = i0; ib < i1; ib += 32 * kU) {
        if (ib != i0) {
#pragma unroll
            for (int u = 0; u < kU; ++u) raw[u] = load_raw(p.topk_idx, ib + u * 32 + lane, i1);
        }
#pragma unroll
        for (int u = 0; u < kU; ++u) {
            if (ib + u * 32 >= i1) break;  // warp-uniform
            const int i = ib + u * 32 + lane;
            const int e = to_key(p, raw[u], i);
            const uint32_t peers = warp_match(e < 0 ? E : e, ebits);
            int local = 0;
            if (e >= 0) local = hist_w[w * E + e] + __popc(peers & lanemask_lt());
            __syncwarp();
            if (e >= 0 && lane == __ffs(peers) - 1) hist_w[w * E + e] += __popc(peers);
            __syncwarp();
            if (i < i1) stage[i] = (local << 11) | (e + 1);
            if (want_er) {
                const int key = e >= 0 ? e * span + (i / K) / T - r0 : E * span;
                const uint32_t pk = warp_match(key, erbits);
                if (e >= 0 && lane == __ffs(pk) - 1) atomicAdd(&hist_er[key], __popc(pk));
            }
        }
    }
    if (p.tokens_per_rank || p.is_token_in_rank) {
        for (int g = t0 + lane; g < t1; g += 32) {
            const int64_t *row = p.topk_idx + (int64_t)g * K;
            for (int k = 0; k < K; ++k) {
                const int64_t e = row[k];
                if (e < 0 || e >= p.num_experts) continue;
                const int d = (int)e / p.L;
                bool seen = false;
                for (int k2 = 0; k2 < k && !seen; ++k2) {
                    const int64_t e2 = row[k2];
                    seen = e2 >= 0 && e2 < p.num_experts && (int)e2 / p.L == d;
                }
                if (seen) continue;
                atomicAdd(&tok_rank[d], 1);
                if (p.is_token_in_rank) p.is_token_in_rank[(int64_t)g * R + d] = 1;
            }
        }
    }
    __syncthreads();
    // per key: exclusive prefix over the CTA's warps (kept); the CTA total to global
    for (int e = tid; e < E; e += NT) {
        int s = 0;
        for (int ww = 0; ww < NW; ++ww) {
            const int v = hist_w[ww * E + e];
            hist_w[ww * E + e] = s;
            s += v;
        }
        p.cta_hist[(int64_t)c * E + e] = s;
    }
    // the per-rank and per-(expert, rank) counts are zeroed here, in slices,
    // and accumulated after the barrier
    if (p.tokens_per_rank && c == 0)
        for (int d = tid; d < R; d += NT) p.tokens_per_rank[d] = 0;
    if (want_er) {
        const int64_t n = (int64_t)E * R, sl = (n + C - 1) / C;
        for (int64_t j = c * sl + tid; j < min(n, (c + 1) * sl); j += NT) p.cnt_er[j] = 0;
    }
    if (!grid_barrier(p.grid_bar, (uint32_t)C, &bar_ok)) {
        if (tid == 0) {
            atomicOr(p.status, kStatusTimeout);
            grid_depart(p.grid_bar, (uint32_t)C, 1u);
        }
        return;
    }
    if (p.tokens_per_rank)
        for (int d = tid; d < R; d += NT)
            if (tok_rank[d] != 0) atomicAdd(&p.tokens_per_rank[d], tok_rank[d]);
    if (want_er)
        for (int j = tid; j < E * span; j += NT)
            if (hist_er[j] != 0) atomicAdd(&p.cnt_er[(j / span) * R + r0 + j % span], hist_er[j]);

    // ---------------- scan of the keys this CTA owns
    // one warp per owned key: lane l takes CTAs [l*per, (l+1)*per) (all its
    // loads in flight at once), a shuffle scan over the lanes gives each
    // slice its start; the same warp then turns the key's per-rank counts
    // into offsets
    {
        const int ke0 = (int)((int64_t)c * E / C), ke1 = (int)((int64_t)(c + 1) * E / C);
        const int per = (C + 31) / 32;  // CTAs per lane: at most 8 up to 256 CTAs, 16 up to 512
        for (int e = ke0 + w; e < ke1; e += NW) {
            int v[8];
            int local = 0;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int cc = lane * per + j;
                v[j] = (j < per && cc < C) ? __ldcg(&p.cta_hist[(int64_t)cc * E + e]) : 0;
                local += v[j];
            }
            for (int j = 8; j < per; ++j) {  // more than 256 CTAs
                const int cc = lane * per + j;
                if (cc < C) local += __ldcg(&p.cta_hist[(int64_t)cc * E + e]);
            }
            int incl = local;
#pragma unroll
            for (int d = 1; d < 32; d <<= 1) {
                const int y = __shfl_up_sync(0xFFFFFFFFu, incl, d);
                if (lane >= d) incl += y;
            }
            int run = incl - local;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int cc = lane * per + j;
                if (j < per && cc < C) p.cta_hist[(int64_t)cc * E + e] = run;
                run += v[j];
            }
            for (int j = 8; j < per; ++j) {
                const int cc = lane * per + j;
                if (cc < C) {
                    const int x = __ldcg(&p.cta_hist[(int64_t)cc * E + e]);
                    p.cta_hist[(int64_t)cc * E + e] = run;
                    run += x;
                }
            }
            const int total = __shfl_sync(0xFFFFFFFFu, incl, 31);
            if (lane == 0) {
                const int n = (int)min((int64_t)total, p.cap);
                p.tokens_per_expert[e] = n;
                if (p.user_tokens_per_expert) p.user_tokens_per_expert[e] = n;
                if (p.layout == kLayoutPadded) p.base[e] = (int64_t)e * p.cap;
            }
        }
    }
    if (!grid_barrier(p.grid_bar, 2u * (uint32_t)C, &bar_ok)) {
        if (tid == 0) {
            atomicOr(p.status, kStatusTimeout);
            grid_depart(p.grid_bar, (uint32_t)C, 0u);
        }
        return;
    }
    if (want_er) {  // the (expert, rank) counts are complete: offsets over the source ranks
        const int ke0 = (int)((int64_t)c * E / C), ke1 = (int)((int64_t)(c + 1) * E / C);
        for (int e = ke0 + w; e < ke1; e += NW) {
            int rrun = 0;
            for (int rr = 0; rr < R; rr += 32) {
                const int r = rr + lane;
                const int cv = r < R ? __ldcg(&p.cnt_er[e * R + r]) : 0;
                int x = cv;
#pragma unroll
                for (int d = 1; d < 32; d <<= 1) {
                    const int y = __shfl_up_sync(0xFFFFFFFFu, x, d);
                    if (lane >= d) x += y;
                }
                if (r < R) p.off_er[e * R + r] = rrun + x - cv;
                rrun += __shfl_sync(0xFFFFFFFFu, x, 31);
            }
        }
    }

    // ---------------- write
    // pre[e] = first row of key e for this CTA's entries: base + lower CTAs
    {
        const int chunk = (E + NT - 1) / NT;
        const int e_lo = min(E, tid * chunk), e_hi = min(E, e_lo + chunk);
        for (int e = e_lo; e < e_hi; ++e) pre[e] = __ldcg(&p.cta_hist[(int64_t)c * E + e]);  // in flight during the scan
        int local = 0;
        if (p.layout != kLayoutPadded)
            for (int e = e_lo; e < e_hi; ++e) local += __ldcg(&p.tokens_per_expert[e]);
        int total;
        int run = block_exclusive_scan<NT>(local, scan, &total);
        for (int e = e_lo; e < e_hi; ++e) {
            const int64_t b = p.layout == kLayoutPadded ? (int64_t)e * p.cap : (int64_t)run;
            if (p.layout != kLayoutPadded) {
                run += __ldcg(&p.tokens_per_expert[e]);
                if (c == 0) p.base[e] = b;
            }
            hist_er[e] = (int32_t)b;  // the (e, r) counts are done with: reuse for the bases
        }
    }
    __syncthreads();
    const int cap = (int)min(p.cap, (int64_t)0x7FFFFFFF);
    for (int i = i0 + lane; i < i1; i += 32) {
        const int v = stage[i];
        const int e = (v & 2047) - 1;
        int32_t s = -1;
        if (e >= 0) {
            const int pos = pre[e] + hist_w[w * E + e] + (v >> 11);
            if (pos < cap) {
                s = hist_er[e] + pos;
                p.src_info[s] = i;
                if (p.recv_topk_idx != nullptr) {  // rank mode: the token's experts on rank e
                    const int g0 = (i / K) * K;
                    for (int k2 = 0; k2 < K; ++k2) {
                        const int64_t e2 = __ldg(p.topk_idx + g0 + k2);
                        const bool on = e2 >= 0 && e2 < p.num_experts && (int)e2 / p.L == e;
                        p.recv_topk_idx[(int64_t)s * K + k2] = on ? (int)e2 - e * p.L : -1;
                        if (p.recv_topk_weights != nullptr)
                            p.recv_topk_weights[(int64_t)s * K + k2] =
                                on ? (p.topk_weights != nullptr ? __ldg(p.topk_weights + g0 + k2) : 1.0f) : 0.0f;
                    }
                }
            } else {
                atomicOr(p.status, kStatusCapacity);
            }
        }
        p.slot[i] = s;
    }
    if (tid == 0) grid_depart(p.grid_bar, (uint32_t)C, 0u);
}

size_t grid_smem(int E, int R, int span, int NT) {
    const int hist_er = E * span > E ? E * span : E;  // reused for the bases in the write phase
    return ((size_t)(NT / 32) * E + R + (size_t)hist_er + E + NT / 32 + 1) * sizeof(int32_t);
}

void grid_init() {
    int dev = 0, optin = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    cudaFuncSetAttribute(layout_grid_kernel<512>, cudaFuncAttributeMaxDynamicSharedMemorySize, optin - 64);
    cudaFuncSetAttribute(layout_grid_kernel<1024>, cudaFuncAttributeMaxDynamicSharedMemorySize, optin - 64);
    cudaGetLastError();
}

}  // namespace

size_t layout_smem_bytes(int E, int R, int threads, int cluster_size) {
    return smem_words(E, R, threads, cluster_size) * sizeof(int32_t);
}

bool layout_pick_shape(int E, int R, int *cluster_size, int *threads, bool many_entries) {
    static const int cls[] = {16, 8, 4, 2, 1};
    grid_init();
    for (int cl : cls) {
        // 512 threads measured fastest at the low-latency sizes (32K entries);
        // from ~64K entries on, 1024 threads hide more of each warp's latency
        // (262K entries: 27 vs 31 µs, 524K: 50 vs 60 µs)
        if (many_entries && fits<1024>(E, R, cl)) { *cluster_size = cl; *threads = 1024; return true; }
        if (fits<512>(E, R, cl)) { *cluster_size = cl; *threads = 512; return true; }
        if (fits<1024>(E, R, cl)) { *cluster_size = cl; *threads = 1024; return true; }
        if (fits<256>(E, R, cl)) { *cluster_size = cl; *threads = 256; return true; }
    }
    return false;
}

cudaError_t launch_layout_grid(LayoutParams p, int ctas, cudaStream_t stream) {
    const int64_t N = p.N;
    if (N <= 0 || ctas < 1 || ctas > 512 || p.grid_bar == nullptr) return cudaErrorInvalidValue;
    const int NT = N * p.K >= kGridBigEntries ? 1024 : 512;
    // tokens per CTA; a warp's entries are packed into 20 bits until the write phase
    int64_t tpc = (N + ctas - 1) / ctas;
    if (tpc * p.K >= (int64_t(1) << 20)) return cudaErrorInvalidConfiguration;
    const int C = (int)((N + tpc - 1) / tpc);
    p.grid_ctas = C;
    p.grid_tpc = (int)tpc;
    p.staged = 0;
    p.er_span = 0;
    if (p.cnt_er != nullptr) {
        const int64_t span = p.T > 0 ? (tpc + p.T - 1) / p.T + 1 : 1;
        p.er_span = (int)(span < p.R ? span : p.R);
    }
    const size_t smem = grid_smem(p.E, p.R, p.er_span, NT);
    if (smem > kMaxSmem) return cudaErrorInvalidConfiguration;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;  // every CTA resident: the grid barriers end
    attr[0].val.cooperative = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.stream = stream;
    cfg.gridDim = dim3((unsigned)C, 1, 1);
    cfg.blockDim = dim3(NT, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = NT == 1024 ? cudaLaunchKernelEx(&cfg, layout_grid_kernel<1024>, p)
                               : cudaLaunchKernelEx(&cfg, layout_grid_kernel<512>, p);
    if (e == cudaErrorCooperativeLaunchTooLarge) return cudaErrorInvalidConfiguration;
    return e;
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
