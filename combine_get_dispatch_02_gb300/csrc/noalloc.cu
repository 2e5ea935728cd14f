// ep_dispatch_noalloc: the dispatch (layout kernel + scatter kernel) with all
// of its intermediate state in one statically allocated device array.
//
// The regular path keeps that state (receive row of every entry, first row
// and count of every expert, the device status word) in buffers that
// ep_create / ep_handle_create obtain with cudaMalloc.  Some callers cannot
// call cudaMalloc: runtimes that hand every byte of device memory to their
// own allocator up front (a cudaMalloc of theirs would fail or steal from
// that pool), plugins that may only touch the memory they are given, and
// code on a latency-critical path where a cudaMalloc could synchronise the
// device.  For them this entry point takes only the inputs and outputs and
// keeps the rest in g_noalloc_scratch below, which the CUDA module of
// libep.so holds on every GPU that loads the library until the process
// exits (about 4.3 MB).
//
// Limits (calls beyond them return EP_ERR_UNSUPPORTED and enqueue nothing):
//   R * tokens_per_rank * K  <= 65536 entries
//   receive rows (ep_recv_rows) <= 1048576
//   num_experts <= 1024
// Every call shares the array: two calls whose work overlaps on the GPU (on
// different streams, or the same call on two threads) race and corrupt each
// other's layout.  Each call clears the status word it uses before its
// kernels run; the rest of the array is fully rewritten before it is read.
#include <mutex>

#include <cuda_runtime.h>

#include "ep.h"
#include "ep_internal.cuh"

namespace {

constexpr int64_t kMaxEntries = 65536;
constexpr int64_t kMaxRows = int64_t(1) << 20;
constexpr int kMaxExperts = 1024;

constexpr size_t kOffSlot = 0;                                  // int32 [kMaxEntries]
constexpr size_t kOffSrcInfo = kOffSlot + kMaxEntries * 4;      // int32 [kMaxRows]
constexpr size_t kOffBase = kOffSrcInfo + kMaxRows * 4;         // int64 [kMaxExperts]
constexpr size_t kOffCount = kOffBase + kMaxExperts * 8;        // int32 [kMaxExperts]
constexpr size_t kOffStatus = kOffCount + kMaxExperts * 4;      // uint32
constexpr size_t kScratchBytes = kOffStatus + 256;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

// Per-device set-up: the device address of g_noalloc_scratch (host code may
// not use the symbol itself as an address), the SM count, resident blocks of
// the dispatch kernels and the layout kernel's shape for the last (E, R).
// The address is looked up again on every call: after a cudaDeviceReset the
// module is loaded anew and the array may sit elsewhere, and then the whole
// set-up (kernel attributes included) is repeated.
struct DeviceSetup {
    bool ready;
    unsigned char *scratch;
    int num_sms;
    int bps_bf16, bps_fp8;
    int shape_E, shape_R, cluster, threads;
};
constexpr int kMaxDevices = 64;
DeviceSetup g_setup[kMaxDevices];
std::mutex g_setup_mutex;

bool aligned(const void *p, size_t a) { return ((uintptr_t)p % a) == 0; }

}  // namespace

extern "C" ep_status ep_dispatch_noalloc(const ep_config *cfg, const void *d_x, const int64_t *d_topk_idx,
                                         int32_t tokens_per_rank, int32_t use_fp8, void *d_recv_x,
                                         float *d_recv_scales, int32_t *d_recv_count, void *stream) {
    const ep_status cs = ep_config_check(cfg);
    if (cs != EP_OK) return cs;
    const ep_config c = *cfg;
    if (tokens_per_rank < 0 || tokens_per_rank > c.max_tokens_per_rank) return EP_ERR_INVALID_ARG;
    if (use_fp8 != 0 && use_fp8 != 1) return EP_ERR_INVALID_ARG;
    if (use_fp8 && c.hidden % 128 != 0) return EP_ERR_UNSUPPORTED;
    int64_t rows = 0;
    ep_recv_rows(cfg, &rows);
    const int64_t N = (int64_t)c.num_ranks * tokens_per_rank;
    if (N * c.topk > kMaxEntries || rows > kMaxRows || c.num_experts > kMaxExperts) return EP_ERR_UNSUPPORTED;
    if (N > 0 && (d_x == nullptr || d_topk_idx == nullptr || d_recv_x == nullptr ||
                  (use_fp8 && d_recv_scales == nullptr)))
        return EP_ERR_INVALID_ARG;
    if (!aligned(d_x, 16) || !aligned(d_recv_x, 16) || !aligned(d_recv_scales, 16) || !aligned(d_recv_count, 4) ||
        !aligned(d_topk_idx, 8))
        return EP_ERR_INVALID_ARG;

    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return EP_ERR_CUDA;
    }
    DeviceSetup s;
    {
        std::lock_guard<std::mutex> lock(g_setup_mutex);
        DeviceSetup &d = g_setup[dev];
        void *ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || ptr == nullptr) {
            cudaGetLastError();
            return EP_ERR_CUDA;
        }
        if (!d.ready || d.scratch != static_cast<unsigned char *>(ptr)) {
            if (cudaDeviceGetAttribute(&d.num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
                cudaGetLastError();
                return EP_ERR_CUDA;
            }
            d.scratch = static_cast<unsigned char *>(ptr);
            d.bps_bf16 = ep::dispatch_blocks_per_sm(false);
            d.bps_fp8 = ep::dispatch_blocks_per_sm(true);
            ep::dispatch_init();
            d.shape_E = d.shape_R = -1;
            d.ready = true;
        }
        if (d.shape_E != c.num_experts || d.shape_R != c.num_ranks) {
            if (!ep::layout_pick_shape(c.num_experts, c.num_ranks, &d.cluster, &d.threads)) return EP_ERR_UNSUPPORTED;
            d.shape_E = c.num_experts;
            d.shape_R = c.num_ranks;
        }
        s = d;
    }

    cudaStream_t st = (cudaStream_t)stream;
    uint32_t *status = reinterpret_cast<uint32_t *>(s.scratch + kOffStatus);
    if (cudaMemsetAsync(status, 0, sizeof(uint32_t), st) != cudaSuccess) {
        cudaGetLastError();
        return EP_ERR_CUDA;
    }
    ep::LayoutParams lp;
    lp.topk_idx = d_topk_idx;
    lp.R = c.num_ranks;
    lp.T = tokens_per_rank;
    lp.K = c.topk;
    lp.E = c.num_experts;
    lp.L = c.num_experts / c.num_ranks;
    lp.num_experts = c.num_experts;
    lp.rank_mode = 0;
    lp.topk_weights = nullptr;
    lp.recv_topk_idx = nullptr;
    lp.recv_topk_weights = nullptr;
    lp.layout = c.layout;
    lp.N = N;
    lp.cap = c.layout == EP_LAYOUT_PADDED ? (int64_t)c.num_ranks * c.max_tokens_per_rank
                                          : (int64_t)c.num_ranks * c.max_tokens_per_rank * c.topk;
    lp.slot = reinterpret_cast<int32_t *>(s.scratch + kOffSlot);
    lp.src_info = reinterpret_cast<int32_t *>(s.scratch + kOffSrcInfo);
    lp.cnt_er = nullptr;
    lp.off_er = nullptr;
    lp.base = reinterpret_cast<int64_t *>(s.scratch + kOffBase);
    lp.tokens_per_expert = reinterpret_cast<int32_t *>(s.scratch + kOffCount);
    lp.user_tokens_per_expert = d_recv_count;
    lp.tokens_per_rank = nullptr;
    lp.is_token_in_rank = nullptr;
    lp.status = status;
    lp.cta_hist = nullptr;  // at most 65536 entries here: always the cluster form
    lp.grid_bar = nullptr;
    const cudaError_t le = ep::launch_layout(lp, s.cluster, s.threads, st);
    if (le != cudaSuccess) {  // the status clear above is already enqueued (harmless)
        cudaGetLastError();
        return le == cudaErrorInvalidConfiguration ? EP_ERR_UNSUPPORTED : EP_ERR_CUDA;
    }
    if (N == 0) return EP_OK;

    ep::DispatchParams dp;
    dp.x = d_x;
    dp.slot = lp.slot;
    dp.recv = d_recv_x;
    dp.recv_scales = d_recv_scales;
    dp.N = N;
    dp.K = c.topk;
    dp.H = c.hidden;
    dp.count_src = nullptr;
    dp.count_dst = nullptr;
    dp.E = c.num_experts;
    int sms = s.num_sms;
    if (c.max_sms > 0 && c.max_sms < sms) sms = c.max_sms;
    // short FP8 rows go to the warp-item kernel (the rule of ep_dispatch)
    const bool short_fp8 = use_fp8 && (c.hidden <= 1024 || (c.hidden <= 2048 && c.topk <= 4));
    dp.row_sms = short_fp8 ? 0 : sms;
    dp.row_bps = 0;
    dp.status = status;
    dp.early_x = 1;  // behind the layout kernel
    dp.token_grid = 0;  // the token kernel by the rule of ep_dispatch (large dispatches on all SMs)
    if (!short_fp8 && ep::token_kernel_rule(N, c.topk, c.hidden, use_fp8 != 0, sms < s.num_sms)) dp.token_grid = N;
    const int cap = sms * (use_fp8 ? s.bps_fp8 : s.bps_bf16);
    const cudaError_t de = ep::launch_dispatch(dp, use_fp8 != 0, cap, /*pdl=*/true, st);
    if (de != cudaSuccess) {
        cudaGetLastError();
        return de == cudaErrorInvalidConfiguration ? EP_ERR_UNSUPPORTED : EP_ERR_CUDA;
    }
    return EP_OK;
}
