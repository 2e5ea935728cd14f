// Combine kernel: top-k weighted gather-reduce of expert outputs back to BF16
// tokens.
//
// Operation: low_latency_combine(hidden_states, topk_idx, topk_weights,
// handle, num_experts) of "如何突破MoE通信瓶颈：DeepEP跨节点优化技术终极指南"
// (section 核心API示例) with the BF16 combine of section 核心优势:
//   out[g, c] = bf16( acc ),  acc = +0;  for k = 0..K-1 ascending, skipping
//   masked entries: acc = fma(w[g,k], y[row(g,k), c], acc)   (fp32)
// so the result is identical to the oracle's bit for bit.
//
// Design: the work item is (token, 256-channel chunk) for one warp, 8
// channels (one 16-byte row segment) per lane.  For each group of up to 8
// entries the warp loads the slots and weights once (lanes 0..7, then
// shuffles) and issues all of the group's 16-byte row loads before the first
// FMA, so each lane has up to 128 bytes in flight; the rows are read-only and
// bypass L1.  One 16-byte store per lane writes the bf16 result.
#include <cuda_bf16.h>

#include "ep_internal.cuh"

namespace ep {

namespace {

constexpr int kThreads = 256;
constexpr int kChunk = 256;  // channels per warp item
constexpr int kGroup = 8;    // entries whose loads are in flight together

__global__ void __launch_bounds__(kThreads) combine_kernel(const CombineParams p) {
    pdl_wait();
    const int lane = threadIdx.x & 31;
    const int64_t warp = ((int64_t)blockIdx.x * kThreads + threadIdx.x) >> 5;
    const int64_t nwarp = ((int64_t)gridDim.x * kThreads) >> 5;
    const int H = p.H, K = p.K;
    const int nch = (H + kChunk - 1) / kChunk;
    const int64_t items = p.N * nch;
    const __nv_bfloat16 *y = static_cast<const __nv_bfloat16 *>(p.y);

    for (int64_t it = warp; it < items; it += nwarp) {
        const int64_t g = it / nch;
        const int c = (int)(it - g * nch) * kChunk + lane * 8;
        const bool act = c < H;
        float acc[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[j] = 0.0f;

        for (int k0 = 0; k0 < K; k0 += kGroup) {
            int32_t s_l = -1;
            float w_l = 1.0f;
            if (lane < kGroup && k0 + lane < K) {
                s_l = p.slot[g * K + k0 + lane];
                if (p.weights != nullptr) w_l = p.weights[g * K + k0 + lane];
            }
            int32_t s[kGroup];
            float w[kGroup];
            uint4 v[kGroup];
#pragma unroll
            for (int j = 0; j < kGroup; ++j) {
                s[j] = __shfl_sync(0xFFFFFFFFu, s_l, j);
                w[j] = __shfl_sync(0xFFFFFFFFu, w_l, j);
            }
#pragma unroll
            for (int j = 0; j < kGroup; ++j) {
                v[j] = make_uint4(0, 0, 0, 0);
                if (act && s[j] >= 0) v[j] = ld_nc_na_v4(y + (int64_t)s[j] * H + c);
            }
#pragma unroll
            for (int j = 0; j < kGroup; ++j) {
                if (s[j] < 0) continue;
                const uint32_t u[4] = {v[j].x, v[j].y, v[j].z, v[j].w};
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    acc[2 * i] = __fmaf_rn(w[j], bf16_lo(u[i]), acc[2 * i]);
                    acc[2 * i + 1] = __fmaf_rn(w[j], bf16_hi(u[i]), acc[2 * i + 1]);
                }
            }
        }
        if (act) {
            uint32_t o[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const __nv_bfloat162 h = __floats2bfloat162_rn(acc[2 * i], acc[2 * i + 1]);
                o[i] = *reinterpret_cast<const uint32_t *>(&h);
            }
            *reinterpret_cast<uint4 *>(static_cast<__nv_bfloat16 *>(p.out) + g * H + c) =
                make_uint4(o[0], o[1], o[2], o[3]);
        }
    }
}

}  // namespace

int combine_blocks_per_sm() {
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, combine_kernel, kThreads, 0) != cudaSuccess) {
        cudaGetLastError();
        return 1;
    }
    return n > 0 ? n : 1;
}

cudaError_t launch_combine(const CombineParams &p, int max_blocks, bool pdl, cudaStream_t stream) {
    const int nch = (p.H + kChunk - 1) / kChunk;
    const int64_t warps = p.N * nch;
    int64_t blocks = (warps + (kThreads / 32) - 1) / (kThreads / 32);
    if (blocks > max_blocks) blocks = max_blocks;
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
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, combine_kernel, p);
}

}  // namespace ep
