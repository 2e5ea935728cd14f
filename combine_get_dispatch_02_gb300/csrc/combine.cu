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
// Design: the work item is (token, CPI 256-channel chunks) for one warp, 8
// channels (one 16-byte row segment) per lane and chunk.  The warp loads the
// token's K slots and weights once (one lane each), keeps the entries that
// received a row (when some are masked, each lane with a row writes it to a
// per-warp list at its rank among them), and for
// each group of 8/CPI of them issues all the group's 16-byte row loads
// before the first FMA, so each lane has up to 8 loads (128 bytes) in
// flight however many entries are masked (CPI follows the most entries a
// token can have rows for: K, or min(K, R) in the rank-deduplicated
// layout).  Rows are read-only and bypass L1.  One 16-byte
// store per lane and chunk writes the bf16 result.
#include <cuda_bf16.h>

#include "ep_internal.cuh"

namespace ep {

namespace {

constexpr int kThreads = 256;
constexpr int kChunk = 256;  // channels per lane-row segment (8 per lane)
constexpr int kLoads = 8;    // 16-byte row loads in flight per lane

// CPI = 256-channel chunks per warp item; entries are taken kLoads / CPI at a
// time (CPI = 2 for more than two entries per token, 4 otherwise).
template <int CPI>
__global__ void __launch_bounds__(kThreads) combine_kernel(const CombineParams p) {
    constexpr int G = kLoads / CPI;  // entries per group
    pdl_wait();
    const int lane = threadIdx.x & 31;
    const int64_t warp = ((int64_t)blockIdx.x * kThreads + threadIdx.x) >> 5;
    const int64_t nwarp = ((int64_t)gridDim.x * kThreads) >> 5;
    const int H = p.H, K = p.K;
    const int nch = (H + kChunk * CPI - 1) / (kChunk * CPI);
    const int64_t items = p.N * nch;
    const __nv_bfloat16 *y = static_cast<const __nv_bfloat16 *>(p.y);
    // per-warp list of a token's entries that have rows (when some are masked)
    __shared__ int32_t list_s[kThreads / 32][32];
    __shared__ float list_w[kThreads / 32][32];
    const int wib = threadIdx.x >> 5;
    const uint32_t all_k = K >= 32 ? 0xFFFFFFFFu : ((1u << K) - 1u);

    for (int64_t it = warp; it < items; it += nwarp) {
        const int64_t g = it / nch;
        const int c0 = (int)(it - g * nch) * kChunk * CPI + lane * 8;
        float acc[CPI][8];
#pragma unroll
        for (int q = 0; q < CPI; ++q)
#pragma unroll
            for (int j = 0; j < 8; ++j) acc[q][j] = 0.0f;

        // the token's entries that received a row, in ascending k, are
        // taken G at a time (masked entries never occupy a load slot)
        int32_t s_all = -1;
        float w_all = 1.0f;
        if (lane < K) {
            s_all = p.slot[g * K + lane];
            if (p.token_major && s_all >= 0) s_all = (int32_t)(g * K + lane);
            if (p.weights != nullptr) w_all = p.weights[g * K + lane];
        }
        const uint32_t valid = __ballot_sync(0xFFFFFFFFu, s_all >= 0);
        const int nv = __popc(valid);
        const bool dense = valid == all_k;  // warp-uniform
        if (!dense) {
            if (s_all >= 0) {
                const int r = __popc(valid & lanemask_lt());
                list_s[wib][r] = s_all;
                list_w[wib][r] = w_all;
            }
            __syncwarp();
        }
        for (int k0 = 0; k0 < nv; k0 += G) {
            int32_t s[G];
            float w[G];
            uint4 v[G][CPI];
#pragma unroll
            for (int j = 0; j < G; ++j) {
                const int n = k0 + j < nv ? k0 + j : 0;
                if (dense) {
                    s[j] = __shfl_sync(0xFFFFFFFFu, s_all, n);
                    w[j] = __shfl_sync(0xFFFFFFFFu, w_all, n);
                } else {
                    s[j] = list_s[wib][n];
                    w[j] = list_w[wib][n];
                }
                if (k0 + j >= nv) s[j] = -1;
            }
#pragma unroll
            for (int j = 0; j < G; ++j)
#pragma unroll
                for (int q = 0; q < CPI; ++q) {
                    v[j][q] = make_uint4(0, 0, 0, 0);
                    const int c = c0 + q * kChunk;
                    if (c < H && s[j] >= 0) v[j][q] = ld_nc_na_v4(y + (int64_t)s[j] * H + c);
                }
#pragma unroll
            for (int j = 0; j < G; ++j) {
                if (s[j] < 0) continue;
#pragma unroll
                for (int q = 0; q < CPI; ++q) {
                    const uint32_t u[4] = {v[j][q].x, v[j][q].y, v[j][q].z, v[j][q].w};
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        acc[q][2 * i] = __fmaf_rn(w[j], bf16_lo(u[i]), acc[q][2 * i]);
                        acc[q][2 * i + 1] = __fmaf_rn(w[j], bf16_hi(u[i]), acc[q][2 * i + 1]);
                    }
                }
            }
        }
        if (!dense) __syncwarp();  // the list is rewritten for the next token
#pragma unroll
        for (int q = 0; q < CPI; ++q) {
            const int c = c0 + q * kChunk;
            if (c >= H) continue;
            uint32_t o[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const __nv_bfloat162 h = __floats2bfloat162_rn(acc[q][2 * i], acc[q][2 * i + 1]);
                o[i] = *reinterpret_cast<const uint32_t *>(&h);
            }
            *reinterpret_cast<uint4 *>(static_cast<__nv_bfloat16 *>(p.out) + g * H + c) =
                make_uint4(o[0], o[1], o[2], o[3]);
        }
    }
}

}  // namespace

namespace {
// chunks per item from the most entries a token can have rows for (two
// chunks measured best from top-3 to top-8, four for top-1 and top-2)
int cpi_for(int valid) { return valid <= 2 ? 4 : 2; }

template <int CPI>
int occupancy() {
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, combine_kernel<CPI>, kThreads, 0) != cudaSuccess) {
        cudaGetLastError();
        return 1;
    }
    return n > 0 ? n : 1;
}
}  // namespace

int combine_cpi_rule(int max_valid) { return cpi_for(max_valid); }

int combine_blocks_per_sm(int max_valid, int cpi) {
    switch (cpi > 0 ? cpi : cpi_for(max_valid)) {
        case 4: return occupancy<4>();
        case 2: return occupancy<2>();
        default: return occupancy<1>();
    }
}

cudaError_t launch_combine(const CombineParams &p, int max_blocks, bool pdl, cudaStream_t stream) {
    const int cpi = p.cpi > 0 ? p.cpi : cpi_for(p.max_valid);
    const int nch = (p.H + kChunk * cpi - 1) / (kChunk * cpi);
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
    switch (cpi) {
        case 4: return cudaLaunchKernelEx(&cfg, combine_kernel<4>, p);
        case 2: return cudaLaunchKernelEx(&cfg, combine_kernel<2>, p);
        default: return cudaLaunchKernelEx(&cfg, combine_kernel<1>, p);
    }
}

}  // namespace ep
