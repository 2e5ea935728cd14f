// Send rows of the rank-deduplicated transport: the position of every
// carried token in a send buffer ordered by (source rank, destination rank,
// token), so that what source rank r sends to rank d is one contiguous run.
//
// The receive that needs no SM ("如何突破MoE通信瓶颈：DeepEP跨节点优化技术终极指南",
// section 技术解析, 通信-计算重叠技术: hook-based overlap occupying no SM;
// the DeepTech announcement of DeepEP, 010bt.com: normal kernels forward
// tokens per destination domain) then moves each run with one copy-engine
// copy: the rows rank d receives are its tokens in ascending global token
// g = r*T + t, so the run from source r is contiguous on the receive side
// too, starting at base[d] + off_er[d][r].
//
// One kernel, behind the rank layout (programmatic dependent launch): every
// CTA first turns the per-(destination, source) counts into the send
// offsets of all R*R runs (an exclusive scan in source-major order, in
// shared memory), then maps its share of the entries:
//   send_slot[i] = send_off[r][d] + (slot[i] - base[d] - off_er[d][r])
// for the entry i = g*K + k that carries token g to rank d = expert / L,
// r = g / T; -1 for every other entry.
#include "ep_internal.cuh"

namespace ep {

namespace {

constexpr int kThreads = 1024;

__global__ void __launch_bounds__(kThreads) rank_send_slot_kernel(const RankSendParams p) {
    __shared__ int32_t soff[kRankRunsMaxRanks * kRankRunsMaxRanks];
    __shared__ int32_t warp_sum[kThreads / 32];
    // the cast into the send buffer may start loading rows now; it waits for
    // this kernel before it reads a send slot
    pdl_launch_dependents();
    pdl_wait();  // counts, offsets and slots of the layout kernel
    const int R = p.R, RR = R * R, t = threadIdx.x, lane = t & 31, w = t >> 5;
    // v = tokens source r = t / R carries to d = t % R (source-major order)
    const int v = t < RR ? p.cnt_er[(t % R) * R + t / R] : 0;
    int x = v;
#pragma unroll
    for (int s = 1; s < 32; s <<= 1) {
        const int y = __shfl_up_sync(0xFFFFFFFFu, x, s);
        if (lane >= s) x += y;
    }
    if (lane == 31) warp_sum[w] = x;
    __syncthreads();
    if (w == 0) {
        const int s0 = warp_sum[lane];
        int incl = s0;
#pragma unroll
        for (int s = 1; s < 32; s <<= 1) {
            const int y = __shfl_up_sync(0xFFFFFFFFu, incl, s);
            if (lane >= s) incl += y;
        }
        warp_sum[lane] = incl - s0;
    }
    __syncthreads();
    if (t < RR) soff[t] = warp_sum[w] + x - v;
    __syncthreads();

    const int64_t NK = p.N * p.K;
    for (int64_t i = (int64_t)blockIdx.x * kThreads + t; i < NK; i += (int64_t)gridDim.x * kThreads) {
        const int32_t s = p.slot[i];
        int32_t out = -1;
        if (s >= 0) {  // a carrying entry: its expert id is valid
            const int d = (int)(p.topk_idx[i] / p.L);
            const int r = (int)((i / p.K) / p.T);
            out = soff[r * R + d] + (s - (int32_t)p.base[d] - p.off_er[d * R + r]);
        }
        p.send_slot[i] = out;
    }
}

}  // namespace

cudaError_t launch_rank_send_slots(const RankSendParams &p, int sms, cudaStream_t stream) {
    if (p.R < 1 || p.R > kRankRunsMaxRanks) return cudaErrorInvalidConfiguration;
    const int64_t NK = p.N * p.K;
    int64_t blocks = (NK + kThreads - 1) / kThreads;
    if (blocks > sms) blocks = sms;
    if (blocks < 1) blocks = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)blocks, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, rank_send_slot_kernel, p);
}

}  // namespace ep
