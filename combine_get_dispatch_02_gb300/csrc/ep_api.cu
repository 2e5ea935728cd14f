// Host side of libep.so: the C ABI declared in include/ep.h — argument checks,
// context / handle management, kernel launches and the copy-engine copies of
// the rank transport.  No call here synchronises the host except
// ep_get_device_status, ep_autotune and the first use of a new rank
// layout's run sizes (ep_rank_dispatch_recv / ep_rank_combine_send /
// ep_rank_runs), and none allocates except ep_create / ep_handle_create /
// ep_autotune, so a dispatch + combine sequence can be captured in a CUDA
// graph.
#include <limits.h>
#include <stdlib.h>
#include <string.h>

#include <algorithm>
#include <vector>

#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>

#include "ep.h"
#include "ep_internal.cuh"

namespace {
constexpr int kCeStreams = 2;  // device wire: copies spread over two streams (measured: 1 stream 2.5,
                               // 2 streams 3.4 TB/s of 29 MB copies)
}

struct ep_ctx {
    ep_config cfg;
    int device;
    int num_sms;
    int64_t rows;
    uint32_t *d_status;
    int layout_cluster;
    int layout_threads;
    int layout_cluster_many;  // shape for layouts of kLayoutManyEntries entries or more
    int layout_threads_many;
    int dispatch_bps_bf16;
    int dispatch_bps_fp8;
    int combine_bps;       // resident combine CTAs per SM, expert layout
    int combine_bps_rank;  // and rank-deduplicated layout
    int identity_bps_bf16;
    int identity_bps_fp8;
    int64_t l2_bytes;
    ep_tuning tune;        // launch shapes set by ep_set_tuning / ep_autotune (0: built-in rules)
    int combine_bps_tuned; // resident combine CTAs per SM for tune.combine_chunks
    ep_tune_record tune_log[24];  // the candidates the last ep_autotune timed
    int tune_log_n;
    ep_test_hooks hooks;   // test-only switches (ep_set_test_hooks)
    // copy-engine streams of the rank transport, forked from and joined back
    // into the caller's stream around each call's copies
    cudaStream_t ce_stream[kCeStreams];
    cudaEvent_t ce_fork;
    cudaEvent_t ce_join[kCeStreams];
    cudaEvent_t ce_rank[ep::kRankRunsMaxRanks];  // host wire: source rank r's first leg has landed
};

struct ep_handle {
    ep_ctx *ctx;
    int32_t *slot;
    int32_t *src_info;
    int32_t *cnt_er;
    int32_t *off_er;
    int64_t *base;
    int32_t *tokens_per_expert;
    int32_t tokens_per_rank;  // -1: no layout yet
    int32_t has_rank_ranges;  // cnt_er / off_er hold the current layout's ranges
    int32_t rank_mode;        // the layout is rank-deduplicated (keys are ranks)
    int32_t num_keys;         // experts, or ranks in rank mode
    int32_t *cta_hist;        // grid-form layout: [num_sms][max(E, R)] per-CTA key totals
    // rank transport (ep_rank_dispatch_send): send row of each carrying entry,
    // and the per-(destination, source) run sizes copied to the host
    int32_t *send_slot;       // [R*Tmax*K]
    int32_t *h_runs;          // pinned host [R*R] (R <= kRankRunsMaxRanks), h_runs[d*R + r]
    cudaEvent_t runs_ev;      // recorded after the copy of the run sizes to h_runs
    int32_t runs_state;       // 0: none, 1: copy queued (wait on runs_ev), 2: on the host
    int32_t has_send;         // send_slot / runs belong to the layout held
};

namespace {

bool aligned(const void *p, size_t a) { return ((uintptr_t)p % a) == 0; }

// A new layout in the handle: the rank transport's send rows and runs no
// longer belong to it.  A copy of old run sizes into h_runs may still be
// queued; the host reads h_runs only after the event of a later send, whose
// copy is queued behind it, and ep_handle_destroy waits for it.
void forget_send(ep_handle *h) {
    h->has_send = 0;
    h->runs_state = 0;
}

// NVTX range around each enqueueing call (free unless a profiler is attached)
struct NvtxRange {
    explicit NvtxRange(const char *name) { nvtxRangePushA(name); }
    ~NvtxRange() { nvtxRangePop(); }
};

ep_status check_config(const ep_config *c) {
    if (c == nullptr) return EP_ERR_INVALID_ARG;
    if (c->num_ranks < 1 || c->max_tokens_per_rank < 1 || c->hidden < 1 || c->num_experts < 1 ||
        c->topk < 1 || c->max_sms < 0)
        return EP_ERR_INVALID_ARG;
    if (c->layout != EP_LAYOUT_PADDED && c->layout != EP_LAYOUT_PACKED) return EP_ERR_INVALID_ARG;
    if (c->num_experts % c->num_ranks != 0) return EP_ERR_INVALID_ARG;
    if (c->hidden % 8 != 0) return EP_ERR_INVALID_ARG;
    if (c->num_ranks > 1024 || c->topk > 32 || c->num_experts > 1024 || c->hidden > 65536)
        return EP_ERR_UNSUPPORTED;
    if ((int64_t)c->num_experts * c->num_ranks > 16384) return EP_ERR_UNSUPPORTED;
    const int64_t n = (int64_t)c->num_ranks * c->max_tokens_per_rank;
    if (n * c->topk >= ((int64_t)1 << 31)) return EP_ERR_UNSUPPORTED;
    if (c->layout == EP_LAYOUT_PADDED && n * c->num_experts >= ((int64_t)1 << 31))
        return EP_ERR_UNSUPPORTED;
    return EP_OK;
}

int64_t rows_of(const ep_config *c) {
    const int64_t n = (int64_t)c->num_ranks * c->max_tokens_per_rank;
    return c->layout == EP_LAYOUT_PADDED ? n * c->num_experts : n * c->topk;
}

// Ints of a handle's per-CTA key totals of the grid-form layout (the grid
// barrier's counter follows them).
size_t grid_hist_ints(const ep_ctx *ctx) {
    const ep_config &c = ctx->cfg;
    return (size_t)ctx->num_sms * (c.num_experts > c.num_ranks ? c.num_experts : c.num_ranks);
}

bool on_ctx_device(const ep_ctx *ctx) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    return dev == ctx->device;
}

int grid_cap(const ep_ctx *ctx, int blocks_per_sm) {
    int sms = ctx->num_sms;
    if (ctx->cfg.max_sms > 0 && ctx->cfg.max_sms < sms) sms = ctx->cfg.max_sms;
    return sms * blocks_per_sm;
}

// The layout kernel(s) for p: one cluster (512 threads per CTA, or 1024 from
// kLayoutManyEntries entries on), or the grid form over all SMs from
// kLayoutGridEntries (rank layout: kLayoutGridEntriesRank) entries on.
cudaError_t launch_layout_any(const ep_ctx *ctx, ep::LayoutParams &p, const ep_handle *h, cudaStream_t stream) {
    const int64_t entries = p.N * p.K;
    p.cta_hist = h->cta_hist;
    p.grid_bar = reinterpret_cast<uint32_t *>(h->cta_hist + grid_hist_ints(ctx));
    const int form = ctx->tune.layout_form;
    const bool grid = form == 2 || (form == 0 && entries >= (p.rank_mode ? ep::kLayoutGridEntriesRank
                                                                         : ep::kLayoutGridEntries));
    if (grid && p.N > 0) {
        int sms = ctx->num_sms;
        if (ctx->cfg.max_sms > 0 && ctx->cfg.max_sms < sms) sms = ctx->cfg.max_sms;
        const cudaError_t e = ep::launch_layout_grid(p, sms, stream);
        if (e != cudaErrorInvalidConfiguration) return e;
        cudaGetLastError();  // beyond the grid form's limits: the cluster form decides
    }
    const bool many = entries >= ep::kLayoutManyEntries;
    return ep::launch_layout(p, many ? ctx->layout_cluster_many : ctx->layout_cluster,
                             many ? ctx->layout_threads_many : ctx->layout_threads, stream);
}

ep_status enqueue_layout(ep_ctx *ctx, const int64_t *topk_idx, int32_t T, int32_t *tokens_per_rank,
                         int32_t *user_tokens_per_expert, uint8_t *is_token_in_rank, bool want_ranges,
                         ep_handle *h, cudaStream_t stream) {
    const ep_config &c = ctx->cfg;
    ep::LayoutParams p;
    p.topk_idx = topk_idx;
    p.R = c.num_ranks;
    p.T = T;
    p.K = c.topk;
    p.E = c.num_experts;
    p.L = c.num_experts / c.num_ranks;
    p.num_experts = c.num_experts;
    p.rank_mode = 0;
    p.topk_weights = nullptr;
    p.recv_topk_idx = nullptr;
    p.recv_topk_weights = nullptr;
    p.layout = c.layout;
    p.N = (int64_t)c.num_ranks * T;
    p.cap = c.layout == EP_LAYOUT_PADDED ? (int64_t)c.num_ranks * c.max_tokens_per_rank
                                         : (int64_t)c.num_ranks * c.max_tokens_per_rank * c.topk;
    p.slot = h->slot;
    p.src_info = h->src_info;
    p.cnt_er = want_ranges ? h->cnt_er : nullptr;
    p.off_er = want_ranges ? h->off_er : nullptr;
    p.base = h->base;
    p.tokens_per_expert = h->tokens_per_expert;
    p.user_tokens_per_expert = user_tokens_per_expert;
    p.tokens_per_rank = tokens_per_rank;
    p.is_token_in_rank = is_token_in_rank;
    p.status = ctx->d_status;
    forget_send(h);
    h->tokens_per_rank = -1;  // until the launches are in: a failed one may have overwritten part of the layout
    const cudaError_t err = launch_layout_any(ctx, p, h, stream);
    if (err != cudaSuccess) {
        cudaGetLastError();
        return err == cudaErrorInvalidConfiguration ? EP_ERR_UNSUPPORTED : EP_ERR_CUDA;
    }
    h->tokens_per_rank = T;
    h->has_rank_ranges = want_ranges ? 1 : 0;
    h->rank_mode = 0;
    h->num_keys = c.num_experts;
    return EP_OK;
}

int64_t rank_rows_of(const ep_config *c) {
    const int64_t n = (int64_t)c->num_ranks * c->max_tokens_per_rank;
    const int64_t kr = c->topk < c->num_ranks ? c->topk : c->num_ranks;
    return c->layout == EP_LAYOUT_PADDED ? n * c->num_ranks : n * kr;
}

// The dispatch kernel over tokens [g0, g1) of the handle's layout (g1 > g0).
ep_status enqueue_dispatch(ep_ctx *ctx, const ep_handle *h, const void *x, int64_t g0, int64_t g1, bool fp8,
                           void *recv, float *recv_scales, int32_t *count_dst, bool behind_layout,
                           cudaStream_t st, bool identity_rows = false, const int32_t *slots = nullptr) {
    const ep_config &c = ctx->cfg;
    ep::DispatchParams p;
    p.x = static_cast<const uint16_t *>(x) + g0 * c.hidden;
    p.slot = identity_rows ? nullptr : (slots != nullptr ? slots : h->slot) + g0 * c.topk;
    p.recv = recv;
    p.recv_scales = recv_scales;
    p.N = g1 - g0;
    p.K = identity_rows ? 1 : c.topk;
    p.H = c.hidden;
    p.count_src = h->tokens_per_expert;
    p.count_dst = count_dst;
    p.E = h->num_keys;
    p.row_sms = (c.max_sms > 0 && c.max_sms < ctx->num_sms) ? c.max_sms : ctx->num_sms;
    // the warp-item kernel when tuned so, and by the rule for short FP8 rows
    // (a <= 2 KB row and a 64-byte scale row per bulk copy pair, too few
    // pairs to amortise the row's staging): H <= 1024 at any top-k, and
    // H <= 2048 up to top-4 (sweep medians at H = 2048: 0.88 vs 0.75 of peak
    // at top-2, 0.89 vs 0.83 at top-3; the row kernel wins from top-6 on,
    // 0.92 vs 0.87)
    const int kern = ctx->tune.dispatch_kernel;
    const bool short_fp8 = fp8 && (c.hidden <= 1024 || (c.hidden <= 2048 && c.topk <= 4));
    if (kern == 2 || (kern == 0 && short_fp8)) p.row_sms = 0;
    p.row_bps = ctx->tune.dispatch_ctas_per_sm;
    p.token_grid = 0;
    // the token kernel when tuned so, and by the rule for large dispatches
    // on all SMs (from 64K receive rows)
    const bool limited = p.row_sms < ctx->num_sms;
    const bool token = kern == 3 || (kern == 0 && !short_fp8 && ep::token_kernel_rule(p.N, p.K, c.hidden, fp8, limited));
    if (token && ep::token_kernel_fits(c.hidden, fp8)) {
        // one CTA per token; on an SM budget a grid of that many SMs' worth
        // of CTAs loops over the tokens
        const int nt = (c.hidden / 16 + 31) / 32 * 32;
        const int bps = nt >= 2048 ? 1 : 2048 / nt;
        p.token_grid = p.row_sms < ctx->num_sms ? (int64_t)p.row_sms * bps : p.N;
    }
    p.status = ctx->d_status;
    p.early_x = behind_layout ? 1 : 0;
    const int cap = grid_cap(ctx, fp8 ? ctx->dispatch_bps_fp8 : ctx->dispatch_bps_bf16);
    if (ep::launch_dispatch(p, fp8, cap, /*pdl=*/true, st) != cudaSuccess) {
        cudaGetLastError();
        return EP_ERR_CUDA;
    }
    return EP_OK;
}

// The identity expert over the rows received by entries of tokens [g0, g1).
ep_status enqueue_identity(ep_ctx *ctx, const ep_handle *h, bool fp8, const void *recv, const float *recv_scales,
                           void *y, int64_t g0, int64_t g1, cudaStream_t st) {
    const ep_config &c = ctx->cfg;
    ep::IdentityParams p;
    p.recv = recv;
    p.recv_scales = recv_scales;
    p.slot = h->slot + g0 * c.topk;
    p.n = (g1 - g0) * c.topk;
    p.H = c.hidden;
    p.y = y;
    const int cap = grid_cap(ctx, fp8 ? ctx->identity_bps_fp8 : ctx->identity_bps_bf16);
    if (ep::launch_identity(p, fp8, cap, /*pdl=*/true, st) != cudaSuccess) {
        cudaGetLastError();
        return EP_ERR_CUDA;
    }
    return EP_OK;
}

// The combine kernel over tokens [g0, g1) (g1 > g0).
ep_status enqueue_combine(ep_ctx *ctx, const ep_handle *h, const void *y, const float *w, int64_t g0, int64_t g1,
                          void *out, cudaStream_t st, bool token_major = false, const int32_t *slots = nullptr) {
    const ep_config &c = ctx->cfg;
    ep::CombineParams p;
    p.y = y;
    p.weights = w != nullptr ? w + g0 * c.topk : nullptr;
    p.slot = (slots != nullptr ? slots : h->slot) + g0 * c.topk;
    p.out = static_cast<uint16_t *>(out) + g0 * c.hidden;
    p.N = g1 - g0;
    p.K = c.topk;
    p.H = c.hidden;
    p.max_valid = h->rank_mode ? (c.topk < c.num_ranks ? c.topk : c.num_ranks) : c.topk;
    p.token_major = token_major ? 1 : 0;
    p.cpi = ctx->tune.combine_chunks;
    const int bps = p.cpi > 0 ? ctx->combine_bps_tuned : (h->rank_mode ? ctx->combine_bps_rank : ctx->combine_bps);
    if (ep::launch_combine(p, grid_cap(ctx, bps), /*pdl=*/true, st) != cudaSuccess) {
        cudaGetLastError();
        return EP_ERR_CUDA;
    }
    return EP_OK;
}

// Automatic chunk of ep_round_trip: the most tokens whose receive rows
// (payload, FP8 scales, and the bf16 expert output unless it is written in
// place) fill about 70% of L2, a multiple of 64 tokens and at least 64.
int32_t auto_chunk(const ep_ctx *ctx, bool fp8, bool rank_mode) {
    if (ctx->tune.round_trip_chunk > 0) return ctx->tune.round_trip_chunk;
    const ep_config &c = ctx->cfg;
    const int64_t rows_per_token = rank_mode ? (c.topk < c.num_ranks ? c.topk : c.num_ranks) : c.topk;
    const int64_t row_bytes = fp8 ? (int64_t)c.hidden + c.hidden / 32 + 2 * (int64_t)c.hidden : 2 * (int64_t)c.hidden;
    const int64_t per_token = rows_per_token * row_bytes;
    int64_t chunk = ctx->l2_bytes * 7 / 10 / per_token / 64 * 64;
    if (chunk < 64) chunk = 64;
    return chunk > INT32_MAX ? INT32_MAX : (int32_t)chunk;
}

// SMs of a copy-engine (row mover) launch: num_sms if positive, else the
// context's limit.
int mover_sms(const ep_ctx *ctx, int32_t num_sms) {
    int sms = ctx->num_sms;
    if (ctx->cfg.max_sms > 0 && ctx->cfg.max_sms < sms) sms = ctx->cfg.max_sms;
    if (num_sms > 0 && num_sms < sms) sms = num_sms;
    return sms;
}

ep_status enqueue_move(const ep_ctx *ctx, ep::MoveParams &p, int sms, cudaStream_t st) {
    p.withhold = ctx->hooks.move_withhold_item;
    p.wait_ns = ctx->hooks.move_wait_ns;
    const cudaError_t e = ep::launch_move(p, sms, /*pdl=*/true, st);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return e == cudaErrorInvalidConfiguration ? EP_ERR_UNSUPPORTED : EP_ERR_CUDA;
    }
    return EP_OK;
}

// Dispatch -> identity expert -> combine over chunks of `chunk` tokens (<= 0
// or > N: one chunk) on the handle's layout.
ep_status enqueue_round_trip(ep_ctx *ctx, const ep_handle *h, const void *x, const float *w, bool fp8, void *recv,
                             float *recv_scales, void *y, void *out, int64_t N, int64_t chunk, bool fresh,
                             cudaStream_t st) {
    if (chunk <= 0 || chunk > N) chunk = N;
    for (int64_t g0 = 0; g0 < N; g0 += chunk) {
        const int64_t g1 = g0 + chunk < N ? g0 + chunk : N;
        ep_status s = enqueue_dispatch(ctx, h, x, g0, g1, fp8, recv, recv_scales, nullptr, fresh || g0 > 0, st);
        if (s == EP_OK && (fp8 || y != recv)) s = enqueue_identity(ctx, h, fp8, recv, recv_scales, y, g0, g1, st);
        if (s == EP_OK) s = enqueue_combine(ctx, h, y, w, g0, g1, out, st);
        if (s != EP_OK) return s;
    }
    return EP_OK;
}

// Checks shared by the calls that run on a handle's cached layout over a
// token range: 0 <= g0 <= g1 <= R*T of the layout.
ep_status check_range(const ep_ctx *ctx, const ep_handle *h, int64_t g0, int64_t g1) {
    if (ctx == nullptr || h == nullptr || h->ctx != ctx) return EP_ERR_INVALID_ARG;
    if (h->tokens_per_rank < 0) return EP_ERR_NO_LAYOUT;
    const int64_t N = (int64_t)ctx->cfg.num_ranks * h->tokens_per_rank;
    if (g0 < 0 || g1 < g0 || g1 > N) return EP_ERR_INVALID_ARG;
    if (!on_ctx_device(ctx)) return EP_ERR_INVALID_ARG;
    return EP_OK;
}

// The rank-deduplicated layout (keys are destination ranks); with
// want_ranges also the per-(destination, source rank) counts and offsets
// that the rank transport's runs come from.
ep_status enqueue_rank_layout(ep_ctx *ctx, const int64_t *topk_idx, const float *topk_weights, int32_t T,
                              int32_t *num_tokens_per_rank, int32_t *recv_topk_idx, float *recv_topk_weights,
                              bool want_ranges, ep_handle *h, cudaStream_t stream) {
    const ep_config &c = ctx->cfg;
    ep::LayoutParams p;
    p.topk_idx = topk_idx;
    p.R = c.num_ranks;
    p.T = T;
    p.K = c.topk;
    p.E = c.num_ranks;  // keys are destination ranks
    p.L = c.num_experts / c.num_ranks;
    p.num_experts = c.num_experts;
    p.rank_mode = 1;
    p.topk_weights = topk_weights;
    p.recv_topk_idx = recv_topk_idx;
    p.recv_topk_weights = recv_topk_weights;
    p.layout = c.layout;
    p.N = (int64_t)c.num_ranks * T;
    p.cap = c.layout == EP_LAYOUT_PADDED ? (int64_t)c.num_ranks * c.max_tokens_per_rank : rank_rows_of(&c);
    p.slot = h->slot;
    p.src_info = h->src_info;
    p.cnt_er = want_ranges ? h->cnt_er : nullptr;
    p.off_er = want_ranges ? h->off_er : nullptr;
    p.base = h->base;
    p.tokens_per_expert = h->tokens_per_expert;
    p.user_tokens_per_expert = num_tokens_per_rank;
    p.tokens_per_rank = nullptr;
    p.is_token_in_rank = nullptr;
    p.status = ctx->d_status;
    forget_send(h);
    h->tokens_per_rank = -1;  // as in enqueue_layout
    const cudaError_t err = launch_layout_any(ctx, p, h, stream);
    if (err != cudaSuccess) {
        cudaGetLastError();
        return err == cudaErrorInvalidConfiguration ? EP_ERR_UNSUPPORTED : EP_ERR_CUDA;
    }
    h->tokens_per_rank = T;
    h->has_rank_ranges = want_ranges ? 1 : 0;
    h->rank_mode = 1;
    h->num_keys = c.num_ranks;
    return EP_OK;
}

// Runs of the rank transport, [r*R + d]: tokens source r carries to rank d,
// and the first send / receive row of each run.
struct RankRuns {
    std::vector<int64_t> cnt, send_off, recv_off;
    int64_t send_rows = 0;
};

// The run sizes on the host: the first use after a new layout waits for the
// copy of the counts that ep_rank_dispatch_send queued (a host
// synchronisation on the end of that send), later uses read them directly.
ep_status rank_runs(const ep_ctx *ctx, ep_handle *h, RankRuns *o) {
    if (!h->has_send || h->runs_state == 0 || h->tokens_per_rank < 0) return EP_ERR_NO_LAYOUT;
    if (h->runs_state == 1) {
        if (cudaEventSynchronize(h->runs_ev) != cudaSuccess) {
            cudaGetLastError();
            return EP_ERR_CUDA;
        }
        h->runs_state = 2;
    }
    const ep_config &c = ctx->cfg;
    const int R = c.num_ranks;
    o->cnt.assign((size_t)R * R, 0);
    o->send_off.assign((size_t)R * R, 0);
    o->recv_off.assign((size_t)R * R, 0);
    for (int r = 0; r < R; ++r)
        for (int d = 0; d < R; ++d) o->cnt[(size_t)r * R + d] = h->h_runs[(size_t)d * R + r];
    int64_t acc = 0;
    for (size_t i = 0; i < (size_t)R * R; ++i) {
        o->send_off[i] = acc;
        acc += o->cnt[i];
    }
    o->send_rows = acc;
    int64_t packed = 0;  // packed layout: rank d's rows start after every lower rank's
    for (int d = 0; d < R; ++d) {
        const int64_t base = c.layout == EP_LAYOUT_PADDED ? (int64_t)d * R * c.max_tokens_per_rank : packed;
        int64_t run = base;
        for (int r = 0; r < R; ++r) {
            o->recv_off[(size_t)r * R + d] = run;
            run += o->cnt[(size_t)r * R + d];
        }
        packed += run - base;
    }
    return EP_OK;
}

// One row block that a wire moves: rows of `row` bytes (and of `row2` bytes
// in a second array, e.g. FP8 scales, when row2 > 0).
struct RowArrays {
    const uint8_t *src, *src2;
    uint8_t *dst, *dst2;
    size_t row, row2;
};

cudaError_t copy_rows(const RowArrays &a, int64_t src_row, int64_t dst_row, int64_t n, cudaMemcpyKind kind,
                      cudaStream_t s) {
    cudaError_t e = cudaMemcpyAsync(a.dst + dst_row * a.row, a.src + src_row * a.row, n * a.row, kind, s);
    if (e == cudaSuccess && a.row2 > 0)
        e = cudaMemcpyAsync(a.dst2 + dst_row * a.row2, a.src2 + src_row * a.row2, n * a.row2, kind, s);
    return e;
}

// Device wire: one device-to-device copy per non-empty run (send -> receive
// rows when to_recv, else receive -> send rows), spread over the context's
// copy streams, forked from and joined back into st.  (The CUDA driver
// carries out same-device copies with its own copy kernels on the SMs.)
ep_status wire_device(ep_ctx *ctx, const RankRuns &t, const RowArrays &a, bool to_recv, cudaStream_t st) {
    const int R = ctx->cfg.num_ranks;
    cudaError_t e = cudaEventRecord(ctx->ce_fork, st);
    for (int i = 0; e == cudaSuccess && i < kCeStreams; ++i) e = cudaStreamWaitEvent(ctx->ce_stream[i], ctx->ce_fork, 0);
    int j = 0;
    for (size_t i = 0; e == cudaSuccess && i < (size_t)R * R; ++i) {
        if (t.cnt[i] == 0) continue;
        const int64_t from = to_recv ? t.send_off[i] : t.recv_off[i], to = to_recv ? t.recv_off[i] : t.send_off[i];
        e = copy_rows(a, from, to, t.cnt[i], cudaMemcpyDeviceToDevice, ctx->ce_stream[j++ % kCeStreams]);
    }
    for (int i = 0; e == cudaSuccess && i < kCeStreams; ++i) {
        e = cudaEventRecord(ctx->ce_join[i], ctx->ce_stream[i]);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(st, ctx->ce_join[i], 0);
    }
    if (e != cudaSuccess) {
        cudaGetLastError();
        return EP_ERR_CUDA;
    }
    return EP_OK;
}

// Host wire: the rows cross through the pinned host buffer `stage` (laid out
// like the send buffer: payload rows, then the second array's rows after
// send_rows_max payload rows) on the copy engines only, one leg per
// direction, pipelined per source rank r: stream 0 carries the first leg
// (device -> host), stream 1 the second (host -> device) of rank r once its
// first leg has landed.
//   to_recv (dispatch):  send rows of r (one copy) -> stage, then each run
//                        stage -> receive rows
//   !to_recv (combine):  each run receive rows -> stage, then the send rows
//                        of r (one copy) stage -> send buffer
ep_status wire_host(ep_ctx *ctx, const RankRuns &t, const RowArrays &a, bool to_recv, uint8_t *stage,
                    int64_t send_rows_max, cudaStream_t st) {
    const int R = ctx->cfg.num_ranks;
    RowArrays leg1 = a, leg2 = a;
    uint8_t *stage2 = stage + send_rows_max * (int64_t)a.row;
    leg1.dst = stage;
    leg1.dst2 = stage2;
    leg2.src = stage;
    leg2.src2 = stage2;
    cudaStream_t s1 = ctx->ce_stream[0], s2 = ctx->ce_stream[1 % kCeStreams];
    cudaError_t e = cudaEventRecord(ctx->ce_fork, st);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(s1, ctx->ce_fork, 0);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(s2, ctx->ce_fork, 0);
    for (int r = 0; e == cudaSuccess && r < R; ++r) {
        const size_t r0 = (size_t)r * R;
        int64_t n_r = 0;
        for (int d = 0; d < R; ++d) n_r += t.cnt[r0 + d];
        if (n_r == 0) continue;
        const int64_t first = t.send_off[r0];  // the send rows of r are contiguous
        if (to_recv) {
            e = copy_rows(leg1, first, first, n_r, cudaMemcpyDeviceToHost, s1);
        } else {
            for (int d = 0; e == cudaSuccess && d < R; ++d)
                if (t.cnt[r0 + d] > 0)
                    e = copy_rows(leg1, t.recv_off[r0 + d], t.send_off[r0 + d], t.cnt[r0 + d], cudaMemcpyDeviceToHost, s1);
        }
        if (e == cudaSuccess) e = cudaEventRecord(ctx->ce_rank[r], s1);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(s2, ctx->ce_rank[r], 0);
        if (to_recv) {
            for (int d = 0; e == cudaSuccess && d < R; ++d)
                if (t.cnt[r0 + d] > 0)
                    e = copy_rows(leg2, t.send_off[r0 + d], t.recv_off[r0 + d], t.cnt[r0 + d], cudaMemcpyHostToDevice, s2);
        } else if (e == cudaSuccess) {
            e = copy_rows(leg2, first, first, n_r, cudaMemcpyHostToDevice, s2);
        }
    }
    if (e == cudaSuccess) e = cudaEventRecord(ctx->ce_join[0], s1);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(st, ctx->ce_join[0], 0);
    if (e == cudaSuccess) e = cudaEventRecord(ctx->ce_join[1 % kCeStreams], s2);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(st, ctx->ce_join[1 % kCeStreams], 0);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return EP_ERR_CUDA;
    }
    return EP_OK;
}

// Pinned (page-locked) host memory: what the copy engines read and write
// without a staging copy of the driver's.
bool pinned_host(const void *p) {
    cudaPointerAttributes at;
    if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    return at.type == cudaMemoryTypeHost;
}

}  // namespace

namespace {

void log_candidate(ep_ctx *ctx, int32_t knob, int32_t value, float us) {
    if (ctx->tune_log_n < 24) ctx->tune_log[ctx->tune_log_n++] = ep_tune_record{knob, value, us};
}

// Median CUDA-event time (µs) of `reps` runs of enqueue().  Before each,
// the first half of `flush` (each half twice the L2 size) is written and the
// second half read: the run starts as it would behind kernels that wrote a
// lot (the write-back of their lines is still draining), the usual place of
// a dispatch or combine in a step — measured, the condition that separates
// the launch shapes (a read-only flush hides differences the step shows).
template <typename F>
ep_status median_us(F enqueue, int reps, void *flush, size_t flush_bytes, int sms, cudaStream_t st, float *us) {
    std::vector<cudaEvent_t> ev(2 * (size_t)reps, nullptr);
    ep_status s = EP_OK;
    for (auto &e : ev)
        if (cudaEventCreate(&e) != cudaSuccess) s = EP_ERR_CUDA;
    for (int r = 0; s == EP_OK && r < reps; ++r) {
        if (flush != nullptr && (cudaMemsetAsync(flush, r & 0xFF, flush_bytes / 2, st) != cudaSuccess ||
                                 ep::launch_l2_evict(static_cast<uint8_t *>(flush) + flush_bytes / 2, flush_bytes / 2,
                                                     sms, st) != cudaSuccess))
            s = EP_ERR_CUDA;
        if (s == EP_OK && cudaEventRecord(ev[2 * r], st) != cudaSuccess) s = EP_ERR_CUDA;
        if (s == EP_OK) s = enqueue();
        if (s == EP_OK && cudaEventRecord(ev[2 * r + 1], st) != cudaSuccess) s = EP_ERR_CUDA;
    }
    if (cudaStreamSynchronize(st) != cudaSuccess && s == EP_OK) s = EP_ERR_CUDA;
    std::vector<float> t;
    for (int r = 0; s == EP_OK && r < reps; ++r) {
        float ms = 0.0f;
        if (cudaEventElapsedTime(&ms, ev[2 * r], ev[2 * r + 1]) != cudaSuccess) s = EP_ERR_CUDA;
        t.push_back(ms * 1000.0f);
    }
    for (auto &e : ev)
        if (e != nullptr) cudaEventDestroy(e);
    if (s != EP_OK) {
        cudaGetLastError();
        return s;
    }
    std::sort(t.begin(), t.end());
    *us = t[t.size() / 2];
    return EP_OK;
}

}  // namespace

extern "C" {

const char *ep_status_str(int32_t s) {
    switch (s) {
        case EP_OK: return "ok";
        case EP_ERR_INVALID_ARG: return "invalid argument";
        case EP_ERR_UNSUPPORTED: return "unsupported size";
        case EP_ERR_OOM: return "device allocation failed";
        case EP_ERR_CUDA: return "CUDA error";
        case EP_ERR_BAD_EXPERT: return "expert id outside [-1, num_experts)";
        case EP_ERR_CAPACITY: return "padded expert buffer overflow";
        case EP_ERR_NO_LAYOUT: return "handle holds no layout for these sizes";
        case EP_ERR_TIMEOUT: return "a bounded wait on the device gave up";
        case EP_ERR_TIMEOUT_IN_FLIGHT: return "a bounded wait on the device gave up with copies still in flight";
        default: return "unknown status";
    }
}

ep_status ep_config_check(const ep_config *cfg) { return check_config(cfg); }

ep_status ep_recv_rows(const ep_config *cfg, int64_t *rows) {
    const ep_status s = check_config(cfg);
    if (s != EP_OK) return s;
    if (rows == nullptr) return EP_ERR_INVALID_ARG;
    *rows = rows_of(cfg);
    return EP_OK;
}

ep_status ep_recv_bytes(const ep_config *cfg, int32_t use_fp8, uint64_t *payload_bytes,
                        uint64_t *scale_bytes) {
    const ep_status s = check_config(cfg);
    if (s != EP_OK) return s;
    if (payload_bytes == nullptr) return EP_ERR_INVALID_ARG;
    if (use_fp8 && cfg->hidden % 128 != 0) return EP_ERR_UNSUPPORTED;
    const uint64_t rows = (uint64_t)rows_of(cfg);
    *payload_bytes = rows * (uint64_t)cfg->hidden * (use_fp8 ? 1u : 2u);
    if (scale_bytes) *scale_bytes = use_fp8 ? rows * (uint64_t)(cfg->hidden / 128) * 4u : 0u;
    return EP_OK;
}

ep_status ep_create(const ep_config *cfg, ep_ctx **out) {
    if (out == nullptr) return EP_ERR_INVALID_ARG;
    *out = nullptr;
    const ep_status s = check_config(cfg);
    if (s != EP_OK) return s;
    ep_ctx *ctx = (ep_ctx *)calloc(1, sizeof(ep_ctx));
    if (ctx == nullptr) return EP_ERR_OOM;
    ctx->cfg = *cfg;
    ctx->rows = rows_of(cfg);
    if (cudaGetDevice(&ctx->device) != cudaSuccess ||
        cudaDeviceGetAttribute(&ctx->num_sms, cudaDevAttrMultiProcessorCount, ctx->device) != cudaSuccess) {
        cudaGetLastError();
        free(ctx);
        return EP_ERR_CUDA;
    }
    if (!ep::layout_pick_shape(cfg->num_experts, cfg->num_ranks, &ctx->layout_cluster, &ctx->layout_threads) ||
        !ep::layout_pick_shape(cfg->num_experts, cfg->num_ranks, &ctx->layout_cluster_many,
                               &ctx->layout_threads_many, true)) {
        free(ctx);
        return EP_ERR_UNSUPPORTED;
    }
    ctx->dispatch_bps_bf16 = ep::dispatch_blocks_per_sm(false);
    ctx->dispatch_bps_fp8 = ep::dispatch_blocks_per_sm(true);
    ctx->combine_bps = ep::combine_blocks_per_sm(cfg->topk);
    ctx->combine_bps_rank = ep::combine_blocks_per_sm(cfg->topk < cfg->num_ranks ? cfg->topk : cfg->num_ranks);
    int l2 = 0;
    if (cudaDeviceGetAttribute(&l2, cudaDevAttrL2CacheSize, ctx->device) != cudaSuccess) {
        cudaGetLastError();
        l2 = 0;
    }
    ctx->l2_bytes = l2;
    ctx->identity_bps_bf16 = ep::identity_blocks_per_sm(false);
    ctx->identity_bps_fp8 = ep::identity_blocks_per_sm(true);
    ep::dispatch_init();
    ep::move_init();
    if (cudaMalloc(&ctx->d_status, sizeof(uint32_t)) != cudaSuccess) {
        cudaGetLastError();
        free(ctx);
        return EP_ERR_OOM;
    }
    if (cudaMemset(ctx->d_status, 0, sizeof(uint32_t)) != cudaSuccess) {
        cudaGetLastError();
        cudaFree(ctx->d_status);
        free(ctx);
        return EP_ERR_CUDA;
    }
    ctx->hooks.move_withhold_item = -1;
    ctx->hooks.move_wait_ns = 0;
    bool ok = cudaEventCreateWithFlags(&ctx->ce_fork, cudaEventDisableTiming) == cudaSuccess;
    for (int i = 0; ok && i < kCeStreams; ++i)
        ok = cudaStreamCreateWithFlags(&ctx->ce_stream[i], cudaStreamNonBlocking) == cudaSuccess &&
             cudaEventCreateWithFlags(&ctx->ce_join[i], cudaEventDisableTiming) == cudaSuccess;
    for (int i = 0; ok && i < ep::kRankRunsMaxRanks; ++i)
        ok = cudaEventCreateWithFlags(&ctx->ce_rank[i], cudaEventDisableTiming) == cudaSuccess;
    if (!ok) {
        cudaGetLastError();
        ep_destroy(ctx);
        return EP_ERR_CUDA;
    }
    *out = ctx;
    return EP_OK;
}

ep_status ep_destroy(ep_ctx *ctx) {
    if (ctx == nullptr) return EP_ERR_INVALID_ARG;
    cudaFree(ctx->d_status);
    if (ctx->ce_fork) cudaEventDestroy(ctx->ce_fork);
    for (int i = 0; i < kCeStreams; ++i) {
        if (ctx->ce_stream[i]) cudaStreamDestroy(ctx->ce_stream[i]);
        if (ctx->ce_join[i]) cudaEventDestroy(ctx->ce_join[i]);
    }
    for (int i = 0; i < ep::kRankRunsMaxRanks; ++i)
        if (ctx->ce_rank[i]) cudaEventDestroy(ctx->ce_rank[i]);
    free(ctx);
    return EP_OK;
}

ep_status ep_handle_create(ep_ctx *ctx, ep_handle **out) {
    if (ctx == nullptr || out == nullptr) return EP_ERR_INVALID_ARG;
    *out = nullptr;
    if (!on_ctx_device(ctx)) return EP_ERR_INVALID_ARG;
    const ep_config &c = ctx->cfg;
    ep_handle *h = (ep_handle *)calloc(1, sizeof(ep_handle));
    if (h == nullptr) return EP_ERR_OOM;
    h->ctx = ctx;
    h->tokens_per_rank = -1;
    h->num_keys = c.num_experts;
    const size_t nk = (size_t)c.num_ranks * c.max_tokens_per_rank * c.topk;
    const size_t er = (size_t)c.num_experts * c.num_ranks;
    bool ok = cudaMalloc(&h->slot, nk * sizeof(int32_t)) == cudaSuccess &&
              cudaMalloc(&h->src_info, (size_t)ctx->rows * sizeof(int32_t)) == cudaSuccess &&
              cudaMalloc(&h->cnt_er, er * sizeof(int32_t)) == cudaSuccess &&
              cudaMalloc(&h->off_er, er * sizeof(int32_t)) == cudaSuccess &&
              cudaMalloc(&h->base, (size_t)c.num_experts * sizeof(int64_t)) == cudaSuccess &&
              cudaMalloc(&h->tokens_per_expert, (size_t)c.num_experts * sizeof(int32_t)) == cudaSuccess &&
              cudaMalloc(&h->cta_hist, (grid_hist_ints(ctx) + 16) * sizeof(int32_t)) == cudaSuccess &&
              cudaMalloc(&h->send_slot, nk * sizeof(int32_t)) == cudaSuccess;
    if (ok && c.num_ranks <= ep::kRankRunsMaxRanks)
        ok = cudaMallocHost(&h->h_runs, (size_t)c.num_ranks * c.num_ranks * sizeof(int32_t)) == cudaSuccess &&
             cudaEventCreateWithFlags(&h->runs_ev, cudaEventDisableTiming) == cudaSuccess;
    if (!ok) {
        cudaGetLastError();
        ep_handle_destroy(h);
        return EP_ERR_OOM;
    }
    // the grid-form layout's barrier counter starts at zero (each launch puts it back)
    if (cudaMemset(h->cta_hist + grid_hist_ints(ctx), 0, 16 * sizeof(int32_t)) != cudaSuccess) {
        cudaGetLastError();
        ep_handle_destroy(h);
        return EP_ERR_CUDA;
    }
    *out = h;
    return EP_OK;
}

ep_status ep_handle_destroy(ep_handle *h) {
    if (h == nullptr) return EP_ERR_INVALID_ARG;
    cudaFree(h->slot);
    cudaFree(h->src_info);
    cudaFree(h->cnt_er);
    cudaFree(h->off_er);
    cudaFree(h->base);
    cudaFree(h->tokens_per_expert);
    cudaFree(h->cta_hist);
    if (h->runs_ev) cudaEventSynchronize(h->runs_ev);  // a queued copy into h_runs lands first
    cudaFree(h->send_slot);
    if (h->h_runs) cudaFreeHost(h->h_runs);
    if (h->runs_ev) cudaEventDestroy(h->runs_ev);
    cudaGetLastError();
    free(h);
    return EP_OK;
}

ep_status ep_handle_get_info(const ep_handle *h, ep_handle_info *out) {
    if (h == nullptr || out == nullptr) return EP_ERR_INVALID_ARG;
    out->tokens_per_rank = h->tokens_per_rank;
    out->num_tokens = h->tokens_per_rank < 0 ? 0 : h->tokens_per_rank * h->ctx->cfg.num_ranks;
    out->rows = h->ctx->rows;
    out->slot = h->slot;
    out->src_info = h->src_info;
    out->cnt_er = h->cnt_er;
    out->off_er = h->off_er;
    out->base = h->base;
    out->tokens_per_expert = h->tokens_per_expert;
    out->has_rank_ranges = h->has_rank_ranges;
    out->rank_mode = h->rank_mode;
    return EP_OK;
}

ep_status ep_get_dispatch_layout(ep_ctx *ctx, const int64_t *d_topk_idx, int32_t tokens_per_rank,
                                 int32_t *d_num_tokens_per_rank, int32_t *d_num_tokens_per_expert,
                                 uint8_t *d_is_token_in_rank, ep_handle *handle, void *stream) {
    NvtxRange nvtx("ep_get_dispatch_layout");
    if (ctx == nullptr || handle == nullptr || handle->ctx != ctx) return EP_ERR_INVALID_ARG;
    if (tokens_per_rank < 0 || tokens_per_rank > ctx->cfg.max_tokens_per_rank) return EP_ERR_INVALID_ARG;
    if (d_topk_idx == nullptr && tokens_per_rank > 0) return EP_ERR_INVALID_ARG;
    if (!aligned(d_topk_idx, 8) || !aligned(d_num_tokens_per_rank, 4) || !aligned(d_num_tokens_per_expert, 4))
        return EP_ERR_INVALID_ARG;
    if (!on_ctx_device(ctx)) return EP_ERR_INVALID_ARG;
    return enqueue_layout(ctx, d_topk_idx, tokens_per_rank, d_num_tokens_per_rank, d_num_tokens_per_expert,
                          d_is_token_in_rank, /*want_ranges=*/true, handle, (cudaStream_t)stream);
}

ep_status ep_rank_recv_rows(const ep_config *cfg, int64_t *rows) {
    const ep_status s = check_config(cfg);
    if (s != EP_OK) return s;
    if (rows == nullptr) return EP_ERR_INVALID_ARG;
    *rows = rank_rows_of(cfg);
    return EP_OK;
}

ep_status ep_get_rank_layout(ep_ctx *ctx, const int64_t *d_topk_idx, const float *d_topk_weights,
                             int32_t tokens_per_rank, int32_t *d_num_tokens_per_rank, int32_t *d_recv_topk_idx,
                             float *d_recv_topk_weights, ep_handle *handle, void *stream) {
    NvtxRange nvtx("ep_get_rank_layout");
    if (ctx == nullptr || handle == nullptr || handle->ctx != ctx) return EP_ERR_INVALID_ARG;
    const ep_config &c = ctx->cfg;
    if (tokens_per_rank < 0 || tokens_per_rank > c.max_tokens_per_rank) return EP_ERR_INVALID_ARG;
    if (d_topk_idx == nullptr && tokens_per_rank > 0) return EP_ERR_INVALID_ARG;
    if (d_recv_topk_weights != nullptr && d_recv_topk_idx == nullptr) return EP_ERR_INVALID_ARG;
    if (!aligned(d_topk_idx, 8) || !aligned(d_topk_weights, 4) || !aligned(d_num_tokens_per_rank, 4) ||
        !aligned(d_recv_topk_idx, 4) || !aligned(d_recv_topk_weights, 4))
        return EP_ERR_INVALID_ARG;
    if (!on_ctx_device(ctx)) return EP_ERR_INVALID_ARG;
    return enqueue_rank_layout(ctx, d_topk_idx, d_topk_weights, tokens_per_rank, d_num_tokens_per_rank,
                               d_recv_topk_idx, d_recv_topk_weights, /*want_ranges=*/false, handle,
                               (cudaStream_t)stream);
}

ep_status ep_dispatch(ep_ctx *ctx, const void *d_x, const int64_t *d_topk_idx, int32_t tokens_per_rank,
                      int32_t use_fp8, ep_handle *handle, void *d_recv_x, float *d_recv_scales,
                      int32_t *d_recv_count, void *stream) {
    NvtxRange nvtx("ep_dispatch");
    if (ctx == nullptr || handle == nullptr || handle->ctx != ctx) return EP_ERR_INVALID_ARG;
    const ep_config &c = ctx->cfg;
    if (tokens_per_rank < 0 || tokens_per_rank > c.max_tokens_per_rank) return EP_ERR_INVALID_ARG;
    if (use_fp8 != 0 && use_fp8 != 1) return EP_ERR_INVALID_ARG;
    if (use_fp8 && c.hidden % 128 != 0) return EP_ERR_UNSUPPORTED;
    const int64_t N = (int64_t)c.num_ranks * tokens_per_rank;
    if (N > 0 && (d_x == nullptr || d_recv_x == nullptr || (use_fp8 && d_recv_scales == nullptr)))
        return EP_ERR_INVALID_ARG;
    if (!aligned(d_x, 16) || !aligned(d_recv_x, 16) || !aligned(d_recv_scales, 16) ||
        !aligned(d_recv_count, 4) || !aligned(d_topk_idx, 8))
        return EP_ERR_INVALID_ARG;
    if (d_topk_idx == nullptr && tokens_per_rank > 0 && handle->tokens_per_rank != tokens_per_rank)
        return EP_ERR_NO_LAYOUT;
    if (!on_ctx_device(ctx)) return EP_ERR_INVALID_ARG;
    cudaStream_t st = (cudaStream_t)stream;

    // With no tokens there is nothing to read: an (empty) layout is computed
    // even when d_topk_idx is NULL.
    const bool fresh = d_topk_idx != nullptr || tokens_per_rank == 0;
    if (fresh) {
        const ep_status s = enqueue_layout(ctx, d_topk_idx, tokens_per_rank, nullptr, d_recv_count, nullptr,
                                           /*want_ranges=*/false, handle, st);
        if (s != EP_OK) return s;
    }
    if (N == 0) {
        if (!fresh && d_recv_count != nullptr &&
            cudaMemcpyAsync(d_recv_count, handle->tokens_per_expert, (size_t)handle->num_keys * sizeof(int32_t),
                            cudaMemcpyDeviceToDevice, st) != cudaSuccess) {
            cudaGetLastError();
            return EP_ERR_CUDA;
        }
        return EP_OK;
    }
    return enqueue_dispatch(ctx, handle, d_x, 0, N, use_fp8 != 0, d_recv_x, d_recv_scales,
                            fresh ? nullptr : d_recv_count, fresh, st);
}

ep_status ep_combine(ep_ctx *ctx, const void *d_y, const float *d_topk_weights, const ep_handle *handle,
                     void *d_out, void *stream) {
    NvtxRange nvtx("ep_combine");
    if (ctx == nullptr || handle == nullptr || handle->ctx != ctx) return EP_ERR_INVALID_ARG;
    if (handle->tokens_per_rank < 0) return EP_ERR_NO_LAYOUT;
    const ep_config &c = ctx->cfg;
    const int64_t N = (int64_t)c.num_ranks * handle->tokens_per_rank;
    if (N == 0) return EP_OK;
    if (d_y == nullptr || d_out == nullptr) return EP_ERR_INVALID_ARG;
    if (!aligned(d_y, 16) || !aligned(d_out, 16) || !aligned(d_topk_weights, 4)) return EP_ERR_INVALID_ARG;
    if (!on_ctx_device(ctx)) return EP_ERR_INVALID_ARG;
    return enqueue_combine(ctx, handle, d_y, d_topk_weights, 0, N, d_out, (cudaStream_t)stream);
}

ep_status ep_dispatch_range(ep_ctx *ctx, const void *d_x, int32_t use_fp8, const ep_handle *handle,
                            int64_t token_begin, int64_t token_end, void *d_recv_x, float *d_recv_scales,
                            void *stream) {
    NvtxRange nvtx("ep_dispatch_range");
    const ep_status s = check_range(ctx, handle, token_begin, token_end);
    if (s != EP_OK) return s;
    if (use_fp8 != 0 && use_fp8 != 1) return EP_ERR_INVALID_ARG;
    if (use_fp8 && ctx->cfg.hidden % 128 != 0) return EP_ERR_UNSUPPORTED;
    if (token_end == token_begin) return EP_OK;
    if (d_x == nullptr || d_recv_x == nullptr || (use_fp8 && d_recv_scales == nullptr)) return EP_ERR_INVALID_ARG;
    if (!aligned(d_x, 16) || !aligned(d_recv_x, 16) || !aligned(d_recv_scales, 16)) return EP_ERR_INVALID_ARG;
    return enqueue_dispatch(ctx, handle, d_x, token_begin, token_end, use_fp8 != 0, d_recv_x, d_recv_scales,
                            nullptr, false, (cudaStream_t)stream);
}

ep_status ep_combine_range(ep_ctx *ctx, const void *d_y, const float *d_topk_weights, const ep_handle *handle,
                           int64_t token_begin, int64_t token_end, void *d_out, void *stream) {
    NvtxRange nvtx("ep_combine_range");
    const ep_status s = check_range(ctx, handle, token_begin, token_end);
    if (s != EP_OK) return s;
    if (token_end == token_begin) return EP_OK;
    if (d_y == nullptr || d_out == nullptr) return EP_ERR_INVALID_ARG;
    if (!aligned(d_y, 16) || !aligned(d_out, 16) || !aligned(d_topk_weights, 4)) return EP_ERR_INVALID_ARG;
    return enqueue_combine(ctx, handle, d_y, d_topk_weights, token_begin, token_end, d_out, (cudaStream_t)stream);
}

ep_status ep_expert_identity(ep_ctx *ctx, const ep_handle *handle, int32_t use_fp8, const void *d_recv_x,
                             const float *d_recv_scales, void *d_y, int64_t token_begin, int64_t token_end,
                             void *stream) {
    NvtxRange nvtx("ep_expert_identity");
    const ep_status s = check_range(ctx, handle, token_begin, token_end);
    if (s != EP_OK) return s;
    if (use_fp8 != 0 && use_fp8 != 1) return EP_ERR_INVALID_ARG;
    if (use_fp8 && ctx->cfg.hidden % 128 != 0) return EP_ERR_UNSUPPORTED;
    if (token_end == token_begin || (!use_fp8 && d_y == d_recv_x)) return EP_OK;
    if (d_recv_x == nullptr || d_y == nullptr || (use_fp8 && d_recv_scales == nullptr)) return EP_ERR_INVALID_ARG;
    if (!aligned(d_recv_x, 16) || !aligned(d_y, 16) || !aligned(d_recv_scales, 16)) return EP_ERR_INVALID_ARG;
    return enqueue_identity(ctx, handle, use_fp8 != 0, d_recv_x, d_recv_scales, d_y, token_begin, token_end,
                            (cudaStream_t)stream);
}

ep_status ep_round_trip(ep_ctx *ctx, const void *d_x, const int64_t *d_topk_idx, int32_t tokens_per_rank,
                        const float *d_topk_weights, int32_t use_fp8, ep_handle *handle, void *d_recv_x,
                        float *d_recv_scales, void *d_y, void *d_out, int32_t chunk_tokens, void *stream) {
    NvtxRange nvtx("ep_round_trip");
    if (ctx == nullptr || handle == nullptr || handle->ctx != ctx) return EP_ERR_INVALID_ARG;
    const ep_config &c = ctx->cfg;
    if (tokens_per_rank < 0 || tokens_per_rank > c.max_tokens_per_rank) return EP_ERR_INVALID_ARG;
    if (use_fp8 != 0 && use_fp8 != 1) return EP_ERR_INVALID_ARG;
    if (use_fp8 && c.hidden % 128 != 0) return EP_ERR_UNSUPPORTED;
    const int64_t N = (int64_t)c.num_ranks * tokens_per_rank;
    if (N > 0 && (d_x == nullptr || d_recv_x == nullptr || d_y == nullptr || d_out == nullptr ||
                  (use_fp8 && d_recv_scales == nullptr)))
        return EP_ERR_INVALID_ARG;
    if (!aligned(d_x, 16) || !aligned(d_recv_x, 16) || !aligned(d_recv_scales, 16) || !aligned(d_y, 16) ||
        !aligned(d_out, 16) || !aligned(d_topk_weights, 4) || !aligned(d_topk_idx, 8))
        return EP_ERR_INVALID_ARG;
    if (d_topk_idx == nullptr && tokens_per_rank > 0 && handle->tokens_per_rank != tokens_per_rank)
        return EP_ERR_NO_LAYOUT;
    if (chunk_tokens < EP_CHUNK_AUTO) return EP_ERR_INVALID_ARG;
    if (!on_ctx_device(ctx)) return EP_ERR_INVALID_ARG;
    cudaStream_t st = (cudaStream_t)stream;
    const bool fresh = d_topk_idx != nullptr || tokens_per_rank == 0;
    if (fresh) {
        const ep_status s = enqueue_layout(ctx, d_topk_idx, tokens_per_rank, nullptr, nullptr, nullptr,
                                           /*want_ranges=*/false, handle, st);
        if (s != EP_OK) return s;
    }
    const int64_t chunk = chunk_tokens == EP_CHUNK_AUTO ? auto_chunk(ctx, use_fp8 != 0, handle->rank_mode != 0)
                                                        : chunk_tokens;
    return enqueue_round_trip(ctx, handle, d_x, d_topk_weights, use_fp8 != 0, d_recv_x, d_recv_scales, d_y, d_out,
                              N, chunk, fresh, st);
}

ep_status ep_dispatch_send(ep_ctx *ctx, const void *d_x, const int64_t *d_topk_idx, int32_t tokens_per_rank,
                           int32_t use_fp8, ep_handle *handle, void *d_send_x, float *d_send_scales, void *stream) {
    NvtxRange nvtx("ep_dispatch_send");
    if (ctx == nullptr || handle == nullptr || handle->ctx != ctx) return EP_ERR_INVALID_ARG;
    const ep_config &c = ctx->cfg;
    if (tokens_per_rank < 0 || tokens_per_rank > c.max_tokens_per_rank) return EP_ERR_INVALID_ARG;
    if (use_fp8 != 0 && use_fp8 != 1) return EP_ERR_INVALID_ARG;
    if (use_fp8 && c.hidden % 512 != 0) return EP_ERR_UNSUPPORTED;
    const int64_t N = (int64_t)c.num_ranks * tokens_per_rank;
    if (N > 0 && (d_x == nullptr || d_send_x == nullptr || (use_fp8 && d_send_scales == nullptr)))
        return EP_ERR_INVALID_ARG;
    if (!aligned(d_x, 16) || !aligned(d_send_x, 16) || !aligned(d_send_scales, 16) || !aligned(d_topk_idx, 8))
        return EP_ERR_INVALID_ARG;
    if (d_topk_idx == nullptr && tokens_per_rank > 0 && handle->tokens_per_rank != tokens_per_rank)
        return EP_ERR_NO_LAYOUT;
    if (!on_ctx_device(ctx)) return EP_ERR_INVALID_ARG;
    cudaStream_t st = (cudaStream_t)stream;
    const bool fresh = d_topk_idx != nullptr || tokens_per_rank == 0;
    if (fresh) {
        const ep_status s = enqueue_layout(ctx, d_topk_idx, tokens_per_rank, nullptr, nullptr, nullptr,
                                           /*want_ranges=*/false, handle, st);
        if (s != EP_OK) return s;
    }
    if (N == 0 || (!use_fp8 && d_send_x == d_x)) return EP_OK;  // BF16 rows are sent from x itself
    return enqueue_dispatch(ctx, handle, d_x, 0, N, use_fp8 != 0, d_send_x, d_send_scales, nullptr, fresh, st,
                            /*identity_rows=*/true);
}

ep_status ep_dispatch_recv(ep_ctx *ctx, const ep_handle *handle, int32_t use_fp8, const void *d_send_x,
                           const float *d_send_scales, void *d_recv_x, float *d_recv_scales, int32_t *d_recv_count,
                           int32_t num_sms, void *stream) {
    NvtxRange nvtx("ep_dispatch_recv");
    if (ctx == nullptr || handle == nullptr || handle->ctx != ctx) return EP_ERR_INVALID_ARG;
    if (handle->tokens_per_rank < 0) return EP_ERR_NO_LAYOUT;
    const ep_config &c = ctx->cfg;
    if (use_fp8 != 0 && use_fp8 != 1) return EP_ERR_INVALID_ARG;
    if (use_fp8 && c.hidden % 512 != 0) return EP_ERR_UNSUPPORTED;
    const int64_t N = (int64_t)c.num_ranks * handle->tokens_per_rank;
    if (N > 0 && (d_send_x == nullptr || d_recv_x == nullptr ||
                  (use_fp8 && (d_send_scales == nullptr || d_recv_scales == nullptr))))
        return EP_ERR_INVALID_ARG;
    if (!aligned(d_send_x, 16) || !aligned(d_recv_x, 16) || !aligned(d_send_scales, 16) ||
        !aligned(d_recv_scales, 16) || !aligned(d_recv_count, 4))
        return EP_ERR_INVALID_ARG;
    if (!on_ctx_device(ctx)) return EP_ERR_INVALID_ARG;
    cudaStream_t st = (cudaStream_t)stream;
    if (N == 0) {
        if (d_recv_count != nullptr &&
            cudaMemcpyAsync(d_recv_count, handle->tokens_per_expert, (size_t)handle->num_keys * sizeof(int32_t),
                            cudaMemcpyDeviceToDevice, st) != cudaSuccess) {
            cudaGetLastError();
            return EP_ERR_CUDA;
        }
        return EP_OK;
    }
    ep::MoveParams p;
    p.src = static_cast<const uint8_t *>(d_send_x);
    p.src_scales = use_fp8 ? reinterpret_cast<const uint8_t *>(d_send_scales) : nullptr;
    p.dst = static_cast<uint8_t *>(d_recv_x);
    p.dst_scales = use_fp8 ? reinterpret_cast<uint8_t *>(d_recv_scales) : nullptr;
    p.slot = handle->slot;
    p.n = N;
    p.K = c.topk;
    p.gather = 0;
    p.row_bytes = use_fp8 ? c.hidden : 2 * c.hidden;
    p.scale_bytes = use_fp8 ? c.hidden / 32 : 0;
    p.ring = 0;
    p.count_src = handle->tokens_per_expert;
    p.count_dst = d_recv_count;
    p.E = handle->num_keys;
    p.status = ctx->d_status;
    return enqueue_move(ctx, p, mover_sms(ctx, num_sms), st);
}

ep_status ep_combine_send(ep_ctx *ctx, const ep_handle *handle, const void *d_y, void *d_send_y, int32_t num_sms,
                          void *stream) {
    NvtxRange nvtx("ep_combine_send");
    if (ctx == nullptr || handle == nullptr || handle->ctx != ctx) return EP_ERR_INVALID_ARG;
    if (handle->tokens_per_rank < 0) return EP_ERR_NO_LAYOUT;
    const ep_config &c = ctx->cfg;
    const int64_t N = (int64_t)c.num_ranks * handle->tokens_per_rank;
    if (N == 0) return EP_OK;
    if (d_y == nullptr || d_send_y == nullptr) return EP_ERR_INVALID_ARG;
    if (!aligned(d_y, 16) || !aligned(d_send_y, 16)) return EP_ERR_INVALID_ARG;
    if (!on_ctx_device(ctx)) return EP_ERR_INVALID_ARG;
    ep::MoveParams p;
    p.src = static_cast<const uint8_t *>(d_y);
    p.src_scales = nullptr;
    p.dst = static_cast<uint8_t *>(d_send_y);
    p.dst_scales = nullptr;
    p.slot = handle->slot;
    p.n = N * c.topk;
    p.K = 1;
    p.gather = 1;
    p.row_bytes = 2 * c.hidden;
    p.scale_bytes = 0;
    p.ring = 0;
    p.count_src = nullptr;
    p.count_dst = nullptr;
    p.E = 0;
    p.status = ctx->d_status;
    return enqueue_move(ctx, p, mover_sms(ctx, num_sms), (cudaStream_t)stream);
}

ep_status ep_combine_recv(ep_ctx *ctx, const ep_handle *handle, const void *d_send_y, const float *d_topk_weights,
                          void *d_out, void *stream) {
    NvtxRange nvtx("ep_combine_recv");
    if (ctx == nullptr || handle == nullptr || handle->ctx != ctx) return EP_ERR_INVALID_ARG;
    if (handle->tokens_per_rank < 0) return EP_ERR_NO_LAYOUT;
    const int64_t N = (int64_t)ctx->cfg.num_ranks * handle->tokens_per_rank;
    if (N == 0) return EP_OK;
    if (d_send_y == nullptr || d_out == nullptr) return EP_ERR_INVALID_ARG;
    if (!aligned(d_send_y, 16) || !aligned(d_out, 16) || !aligned(d_topk_weights, 4)) return EP_ERR_INVALID_ARG;
    if (!on_ctx_device(ctx)) return EP_ERR_INVALID_ARG;
    return enqueue_combine(ctx, handle, d_send_y, d_topk_weights, 0, N, d_out, (cudaStream_t)stream,
                           /*token_major=*/true);
}

ep_status ep_rank_send_rows(const ep_config *cfg, int64_t *rows) {
    const ep_status s = check_config(cfg);
    if (s != EP_OK) return s;
    if (rows == nullptr) return EP_ERR_INVALID_ARG;
    const int64_t n = (int64_t)cfg->num_ranks * cfg->max_tokens_per_rank;
    *rows = n * (cfg->topk < cfg->num_ranks ? cfg->topk : cfg->num_ranks);
    return EP_OK;
}

ep_status ep_rank_dispatch_send(ep_ctx *ctx, const void *d_x, const int64_t *d_topk_idx, const float *d_topk_weights,
                                int32_t tokens_per_rank, int32_t use_fp8, int32_t *d_recv_topk_idx,
                                float *d_recv_topk_weights, ep_handle *handle, void *d_send_x, float *d_send_scales,
                                void *stream) {
    NvtxRange nvtx("ep_rank_dispatch_send");
    if (ctx == nullptr || handle == nullptr || handle->ctx != ctx) return EP_ERR_INVALID_ARG;
    const ep_config &c = ctx->cfg;
    if (c.num_ranks > ep::kRankRunsMaxRanks) return EP_ERR_UNSUPPORTED;
    if (tokens_per_rank < 0 || tokens_per_rank > c.max_tokens_per_rank) return EP_ERR_INVALID_ARG;
    if (use_fp8 != 0 && use_fp8 != 1) return EP_ERR_INVALID_ARG;
    if (use_fp8 && c.hidden % 128 != 0) return EP_ERR_UNSUPPORTED;
    if (d_recv_topk_weights != nullptr && d_recv_topk_idx == nullptr) return EP_ERR_INVALID_ARG;
    const int64_t N = (int64_t)c.num_ranks * tokens_per_rank;
    if (N > 0 && (d_x == nullptr || d_send_x == nullptr || (use_fp8 && d_send_scales == nullptr)))
        return EP_ERR_INVALID_ARG;
    if (!aligned(d_x, 16) || !aligned(d_send_x, 16) || !aligned(d_send_scales, 16) || !aligned(d_topk_idx, 8) ||
        !aligned(d_topk_weights, 4) || !aligned(d_recv_topk_idx, 4) || !aligned(d_recv_topk_weights, 4))
        return EP_ERR_INVALID_ARG;
    const bool fresh = d_topk_idx != nullptr || tokens_per_rank == 0;
    if (!fresh && (!handle->has_send || handle->tokens_per_rank != tokens_per_rank)) return EP_ERR_NO_LAYOUT;
    if (!on_ctx_device(ctx)) return EP_ERR_INVALID_ARG;
    cudaStream_t st = (cudaStream_t)stream;
    if (fresh) {
        ep_status s = enqueue_rank_layout(ctx, d_topk_idx, d_topk_weights, tokens_per_rank, nullptr, d_recv_topk_idx,
                                          d_recv_topk_weights, /*want_ranges=*/true, handle, st);
        if (s != EP_OK) return s;
        ep::RankSendParams rp;
        rp.topk_idx = d_topk_idx;
        rp.slot = handle->slot;
        rp.cnt_er = handle->cnt_er;
        rp.off_er = handle->off_er;
        rp.base = handle->base;
        rp.send_slot = handle->send_slot;
        rp.N = N;
        rp.R = c.num_ranks;
        rp.T = tokens_per_rank;
        rp.K = c.topk;
        rp.L = c.num_experts / c.num_ranks;
        if (N > 0 && ep::launch_rank_send_slots(rp, ctx->num_sms, st) != cudaSuccess) {
            cudaGetLastError();
            handle->tokens_per_rank = -1;
            return EP_ERR_CUDA;
        }
    }
    if (N > 0) {
        const ep_status s = enqueue_dispatch(ctx, handle, d_x, 0, N, use_fp8 != 0, d_send_x, d_send_scales, nullptr,
                                             fresh, st, /*identity_rows=*/false, handle->send_slot);
        if (s != EP_OK) {
            if (fresh) handle->tokens_per_rank = -1;
            return s;
        }
    }
    if (fresh) {  // the run sizes, for the host that issues the wire's copies
        const size_t rr = (size_t)c.num_ranks * c.num_ranks;
        if (cudaMemcpyAsync(handle->h_runs, handle->cnt_er, rr * sizeof(int32_t), cudaMemcpyDeviceToHost, st) !=
                cudaSuccess ||
            cudaEventRecord(handle->runs_ev, st) != cudaSuccess) {
            cudaGetLastError();
            handle->tokens_per_rank = -1;
            return EP_ERR_CUDA;
        }
        handle->runs_state = 1;
        handle->has_send = 1;
    }
    return EP_OK;
}

namespace {
// Checks and run table shared by the two wire calls.
ep_status wire_prologue(ep_ctx *ctx, ep_handle *h, int32_t wire, const void *h_stage, RankRuns *t) {
    if (ctx == nullptr || h == nullptr || h->ctx != ctx) return EP_ERR_INVALID_ARG;
    if (wire != EP_WIRE_DEVICE && wire != EP_WIRE_HOST) return EP_ERR_INVALID_ARG;
    if (!h->has_send || h->tokens_per_rank < 0) return EP_ERR_NO_LAYOUT;
    if (!on_ctx_device(ctx)) return EP_ERR_INVALID_ARG;
    if (wire == EP_WIRE_HOST && (h_stage == nullptr || !aligned(h_stage, 16) || !pinned_host(h_stage)))
        return EP_ERR_INVALID_ARG;
    return rank_runs(ctx, h, t);
}
}  // namespace

ep_status ep_rank_dispatch_recv(ep_ctx *ctx, ep_handle *handle, int32_t use_fp8, const void *d_send_x,
                                const float *d_send_scales, void *d_recv_x, float *d_recv_scales,
                                int32_t *d_recv_count, int32_t wire, void *h_stage, void *stream) {
    NvtxRange nvtx("ep_rank_dispatch_recv");
    if (use_fp8 != 0 && use_fp8 != 1) return EP_ERR_INVALID_ARG;
    if (ctx != nullptr && use_fp8 && ctx->cfg.hidden % 128 != 0) return EP_ERR_UNSUPPORTED;
    if (!aligned(d_send_x, 16) || !aligned(d_recv_x, 16) || !aligned(d_send_scales, 16) ||
        !aligned(d_recv_scales, 16) || !aligned(d_recv_count, 4))
        return EP_ERR_INVALID_ARG;
    RankRuns t;
    ep_status s = wire_prologue(ctx, handle, wire, h_stage, &t);
    if (s != EP_OK) return s;
    const ep_config &c = ctx->cfg;
    if (t.send_rows > 0 && (d_send_x == nullptr || d_recv_x == nullptr ||
                            (use_fp8 && (d_send_scales == nullptr || d_recv_scales == nullptr))))
        return EP_ERR_INVALID_ARG;
    cudaStream_t st = (cudaStream_t)stream;
    if (d_recv_count != nullptr &&
        cudaMemcpyAsync(d_recv_count, handle->tokens_per_expert, (size_t)c.num_ranks * sizeof(int32_t),
                        cudaMemcpyDeviceToDevice, st) != cudaSuccess) {
        cudaGetLastError();
        return EP_ERR_CUDA;
    }
    if (t.send_rows == 0) return EP_OK;
    RowArrays a;
    a.src = static_cast<const uint8_t *>(d_send_x);
    a.dst = static_cast<uint8_t *>(d_recv_x);
    a.row = use_fp8 ? (size_t)c.hidden : 2 * (size_t)c.hidden;
    a.src2 = use_fp8 ? reinterpret_cast<const uint8_t *>(d_send_scales) : nullptr;
    a.dst2 = use_fp8 ? reinterpret_cast<uint8_t *>(d_recv_scales) : nullptr;
    a.row2 = use_fp8 ? (size_t)c.hidden / 32 : 0;
    int64_t rows_max = 0;
    ep_rank_send_rows(&c, &rows_max);
    return wire == EP_WIRE_DEVICE ? wire_device(ctx, t, a, true, st)
                                  : wire_host(ctx, t, a, true, static_cast<uint8_t *>(h_stage), rows_max, st);
}

ep_status ep_rank_combine_send(ep_ctx *ctx, ep_handle *handle, const void *d_y, void *d_send_y, int32_t wire,
                               void *h_stage, void *stream) {
    NvtxRange nvtx("ep_rank_combine_send");
    if (!aligned(d_y, 16) || !aligned(d_send_y, 16)) return EP_ERR_INVALID_ARG;
    RankRuns t;
    ep_status s = wire_prologue(ctx, handle, wire, h_stage, &t);
    if (s != EP_OK) return s;
    if (t.send_rows == 0) return EP_OK;
    if (d_y == nullptr || d_send_y == nullptr) return EP_ERR_INVALID_ARG;
    const ep_config &c = ctx->cfg;
    RowArrays a;
    a.src = static_cast<const uint8_t *>(d_y);
    a.dst = static_cast<uint8_t *>(d_send_y);
    a.row = 2 * (size_t)c.hidden;
    a.src2 = nullptr;
    a.dst2 = nullptr;
    a.row2 = 0;
    int64_t rows_max = 0;
    ep_rank_send_rows(&c, &rows_max);
    cudaStream_t st = (cudaStream_t)stream;
    return wire == EP_WIRE_DEVICE ? wire_device(ctx, t, a, false, st)
                                  : wire_host(ctx, t, a, false, static_cast<uint8_t *>(h_stage), rows_max, st);
}

ep_status ep_rank_combine_recv(ep_ctx *ctx, const ep_handle *handle, const void *d_send_y, void *d_out,
                               void *stream) {
    NvtxRange nvtx("ep_rank_combine_recv");
    if (ctx == nullptr || handle == nullptr || handle->ctx != ctx) return EP_ERR_INVALID_ARG;
    if (!handle->has_send || handle->tokens_per_rank < 0) return EP_ERR_NO_LAYOUT;
    const int64_t N = (int64_t)ctx->cfg.num_ranks * handle->tokens_per_rank;
    if (N == 0) return EP_OK;
    if (d_send_y == nullptr || d_out == nullptr) return EP_ERR_INVALID_ARG;
    if (!aligned(d_send_y, 16) || !aligned(d_out, 16)) return EP_ERR_INVALID_ARG;
    if (!on_ctx_device(ctx)) return EP_ERR_INVALID_ARG;
    return enqueue_combine(ctx, handle, d_send_y, nullptr, 0, N, d_out, (cudaStream_t)stream,
                           /*token_major=*/false, handle->send_slot);
}

ep_status ep_rank_runs(ep_handle *handle, int32_t *run_cnt, int64_t *send_off, int64_t *recv_off) {
    if (handle == nullptr) return EP_ERR_INVALID_ARG;
    if (!on_ctx_device(handle->ctx)) return EP_ERR_INVALID_ARG;
    RankRuns t;
    const ep_status s = rank_runs(handle->ctx, handle, &t);
    if (s != EP_OK) return s;
    for (size_t i = 0; i < t.cnt.size(); ++i) {
        if (run_cnt) run_cnt[i] = (int32_t)t.cnt[i];
        if (send_off) send_off[i] = t.send_off[i];
        if (recv_off) recv_off[i] = t.recv_off[i];
    }
    return EP_OK;
}

ep_status ep_round_trip_auto_chunk(const ep_ctx *ctx, int32_t use_fp8, int32_t rank_layout, int32_t *chunk_tokens) {
    if (ctx == nullptr || chunk_tokens == nullptr) return EP_ERR_INVALID_ARG;
    if (use_fp8 != 0 && use_fp8 != 1) return EP_ERR_INVALID_ARG;
    *chunk_tokens = auto_chunk(ctx, use_fp8 != 0, rank_layout != 0);
    return EP_OK;
}

ep_status ep_get_tuning(const ep_ctx *ctx, ep_tuning *out) {
    if (ctx == nullptr || out == nullptr) return EP_ERR_INVALID_ARG;
    *out = ctx->tune;
    return EP_OK;
}

ep_status ep_set_tuning(ep_ctx *ctx, const ep_tuning *t) {
    if (ctx == nullptr || t == nullptr) return EP_ERR_INVALID_ARG;
    if (t->dispatch_ctas_per_sm < 0 || t->dispatch_ctas_per_sm > 16) return EP_ERR_INVALID_ARG;
    if (t->combine_chunks != 0 && t->combine_chunks != 1 && t->combine_chunks != 2 && t->combine_chunks != 4)
        return EP_ERR_INVALID_ARG;
    if (t->round_trip_chunk < 0) return EP_ERR_INVALID_ARG;
    if (t->dispatch_kernel < 0 || t->dispatch_kernel > 3) return EP_ERR_INVALID_ARG;
    if (t->layout_form < 0 || t->layout_form > 2) return EP_ERR_INVALID_ARG;
    if (!on_ctx_device(ctx)) return EP_ERR_INVALID_ARG;
    ctx->tune = *t;
    ctx->combine_bps_tuned = t->combine_chunks > 0 ? ep::combine_blocks_per_sm(0, t->combine_chunks) : 0;
    return EP_OK;
}


ep_status ep_autotune(ep_ctx *ctx, const void *d_x, const int64_t *d_topk_idx, int32_t tokens_per_rank,
                      const float *d_topk_weights, int32_t use_fp8, void *d_recv_x, float *d_recv_scales, void *d_y,
                      void *d_out, int32_t reps, ep_tuning *out, void *stream) {
    if (ctx == nullptr || out == nullptr) return EP_ERR_INVALID_ARG;
    const ep_config &c = ctx->cfg;
    if (tokens_per_rank < 1 || tokens_per_rank > c.max_tokens_per_rank || reps < 1 || reps > 1000)
        return EP_ERR_INVALID_ARG;
    if (use_fp8 != 0 && use_fp8 != 1) return EP_ERR_INVALID_ARG;
    if (use_fp8 && c.hidden % 128 != 0) return EP_ERR_UNSUPPORTED;
    if (d_x == nullptr || d_topk_idx == nullptr || d_recv_x == nullptr || d_y == nullptr || d_out == nullptr ||
        (use_fp8 && d_recv_scales == nullptr))
        return EP_ERR_INVALID_ARG;
    if (!aligned(d_x, 16) || !aligned(d_recv_x, 16) || !aligned(d_recv_scales, 16) || !aligned(d_y, 16) ||
        !aligned(d_out, 16) || !aligned(d_topk_weights, 4) || !aligned(d_topk_idx, 8))
        return EP_ERR_INVALID_ARG;
    if (!on_ctx_device(ctx)) return EP_ERR_INVALID_ARG;
    cudaStream_t st = (cudaStream_t)stream;
    const bool fp8 = use_fp8 != 0;
    const int64_t N = (int64_t)c.num_ranks * tokens_per_rank;

    ep_handle *h = nullptr;
    ep_status s = ep_handle_create(ctx, &h);
    if (s != EP_OK) return s;
    void *flush = nullptr;
    const size_t flush_bytes = (size_t)(ctx->l2_bytes > 0 ? 4 * ctx->l2_bytes : 0);
    if (flush_bytes > 0 && (cudaMalloc(&flush, flush_bytes) != cudaSuccess ||
                            cudaMemsetAsync(flush, 0, flush_bytes, st) != cudaSuccess)) {
        cudaGetLastError();
        if (flush != nullptr) cudaFree(flush);
        flush = nullptr;  // tune without evicting L2
    }
    const int sms = ctx->num_sms;
    const ep_tuning saved = ctx->tune;
    ep_tuning best = saved;
    ctx->tune_log_n = 0;
    s = enqueue_layout(ctx, d_topk_idx, tokens_per_rank, nullptr, nullptr, nullptr, false, h, st);

    // Each knob: the built-in rule's choice is timed first and kept unless
    // another candidate is at least kMargin faster (the medians of runs that
    // start behind a large write differ by a few per cent from run to run).
    constexpr float kMargin = 0.97f;

    // layout form: the rule's, the cluster and the grid form, each timed as
    // layout + dispatch (the rule's dispatch shape)
    if (s == EP_OK) {
        float best_us = 0.0f;
        for (int j = 0; s == EP_OK && j < 3; ++j) {
            ep_tuning t = best;
            t.layout_form = j;
            s = ep_set_tuning(ctx, &t);
            float us = 0.0f;
            if (s == EP_OK)
                s = median_us(
                    [&] {
                        ep_status e = enqueue_layout(ctx, d_topk_idx, tokens_per_rank, nullptr, nullptr, nullptr,
                                                     false, h, st);
                        return e != EP_OK ? e
                                          : enqueue_dispatch(ctx, h, d_x, 0, N, fp8, d_recv_x, d_recv_scales,
                                                             nullptr, true, st);
                    },
                    reps, flush, flush_bytes, sms, st, &us);
            if (s == EP_OK) log_candidate(ctx, EP_TUNE_LAYOUT_FORM, j, us);
            if (s == EP_OK && (j == 0 || us < kMargin * best_us)) {
                best_us = us;
                best.layout_form = j;
            }
        }
    }
    // dispatch: (kernel, row-kernel CTAs per SM), timed as the common call
    // runs it (layout kernel, then the dispatch behind it); the rule first
    if (s == EP_OK) {
        std::vector<std::pair<int, int>> cands = {{0, 0}};
        if (c.hidden % 512 == 0 && c.hidden <= 16384)
            for (int b = 1; b <= 4; ++b) cands.push_back({1, b});
        cands.push_back({2, 0});
        if (ep::token_kernel_fits(c.hidden, fp8)) cands.push_back({3, 0});
        float best_us = 0.0f;
        for (size_t j = 0; s == EP_OK && j < cands.size(); ++j) {
            ep_tuning t = best;
            t.dispatch_kernel = cands[j].first;
            t.dispatch_ctas_per_sm = cands[j].second;
            s = ep_set_tuning(ctx, &t);
            float us = 0.0f;
            if (s == EP_OK)
                s = median_us(
                    [&] {
                        ep_status e = enqueue_layout(ctx, d_topk_idx, tokens_per_rank, nullptr, nullptr, nullptr,
                                                     false, h, st);
                        return e != EP_OK ? e
                                          : enqueue_dispatch(ctx, h, d_x, 0, N, fp8, d_recv_x, d_recv_scales,
                                                             nullptr, true, st);
                    },
                    reps, flush, flush_bytes, sms, st, &us);
            if (s == EP_OK) log_candidate(ctx, EP_TUNE_DISPATCH, 100 * cands[j].first + cands[j].second, us);
            if (s == EP_OK && (j == 0 || us < kMargin * best_us)) {
                best_us = us;
                best.dispatch_kernel = cands[j].first;
                best.dispatch_ctas_per_sm = cands[j].second;
            }
        }
    }
    // combine: chunks per work item
    if (s == EP_OK) {
        const int rule = ep::combine_cpi_rule(c.topk);
        std::vector<int> cands = {rule};
        for (int v : {1, 2, 4})
            if (v != rule) cands.push_back(v);
        float best_us = 0.0f;
        for (size_t j = 0; s == EP_OK && j < cands.size(); ++j) {
            ep_tuning t = best;
            t.combine_chunks = cands[j];
            s = ep_set_tuning(ctx, &t);
            float us = 0.0f;
            if (s == EP_OK)
                s = median_us([&] { return enqueue_combine(ctx, h, d_y, d_topk_weights, 0, N, d_out, st); }, reps,
                              flush, flush_bytes, sms, st, &us);
            if (s == EP_OK) log_candidate(ctx, EP_TUNE_COMBINE_CHUNKS, cands[j], us);
            if (s == EP_OK && (j == 0 || us < kMargin * best_us)) {
                best_us = us;
                best.combine_chunks = cands[j];
            }
        }
    }
    // round trip: the L2 rule's chunk, half and twice that, and one chunk
    if (s == EP_OK) {
        ep_tuning t = best;
        t.round_trip_chunk = 0;
        s = ep_set_tuning(ctx, &t);
        const int64_t rule = auto_chunk(ctx, fp8, false);
        std::vector<int64_t> cands = {rule >= N ? N : rule, N, rule / 2 / 64 * 64, 2 * rule};
        float best_us = 0.0f;
        bool first = true;
        std::vector<int64_t> done;
        for (int64_t ch : cands) {
            if (s != EP_OK) break;
            if (ch < 64 && ch != N) continue;
            if (ch > N) ch = N;
            if (std::find(done.begin(), done.end(), ch) != done.end()) continue;
            done.push_back(ch);
            float us = 0.0f;
            s = median_us([&] { return enqueue_round_trip(ctx, h, d_x, d_topk_weights, fp8, d_recv_x, d_recv_scales,
                                                          d_y, d_out, N, ch, false, st); },
                          reps, flush, flush_bytes, sms, st, &us);
            const int32_t value = ch >= N ? INT32_MAX : (int32_t)ch;  // INT32_MAX: one chunk
            if (s == EP_OK) log_candidate(ctx, EP_TUNE_ROUND_TRIP_CHUNK, value, us);
            if (s == EP_OK && (first || us < kMargin * best_us)) {
                best_us = us;
                best.round_trip_chunk = value;
                first = false;
            }
        }
    }
    if (flush != nullptr) cudaFree(flush);
    ep_handle_destroy(h);
    if (s == EP_OK) s = ep_set_tuning(ctx, &best);
    else ep_set_tuning(ctx, &saved);
    if (s == EP_OK) *out = best;
    return s;
}

ep_status ep_get_autotune_log(const ep_ctx *ctx, ep_tune_record *records, int32_t capacity, int32_t *count) {
    if (ctx == nullptr || count == nullptr || capacity < 0 || (capacity > 0 && records == nullptr))
        return EP_ERR_INVALID_ARG;
    *count = ctx->tune_log_n;
    for (int i = 0; i < ctx->tune_log_n && i < capacity; ++i) records[i] = ctx->tune_log[i];
    return EP_OK;
}

ep_status ep_get_device_status(ep_ctx *ctx, void *stream) {
    if (ctx == nullptr) return EP_ERR_INVALID_ARG;
    if (!on_ctx_device(ctx)) return EP_ERR_INVALID_ARG;
    uint32_t bits = 0;
    if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess ||
        cudaMemcpy(&bits, ctx->d_status, sizeof bits, cudaMemcpyDeviceToHost) != cudaSuccess ||
        cudaMemset(ctx->d_status, 0, sizeof bits) != cudaSuccess) {
        cudaGetLastError();
        return EP_ERR_CUDA;
    }
    if (bits & ep::kStatusBadExpert) return EP_ERR_BAD_EXPERT;
    if (bits & ep::kStatusCapacity) return EP_ERR_CAPACITY;
    if (bits & ep::kStatusInFlight) return EP_ERR_TIMEOUT_IN_FLIGHT;
    if (bits & ep::kStatusTimeout) return EP_ERR_TIMEOUT;
    return EP_OK;
}

ep_status ep_set_test_hooks(ep_ctx *ctx, const ep_test_hooks *hooks) {
    if (ctx == nullptr || hooks == nullptr) return EP_ERR_INVALID_ARG;
    if (hooks->move_withhold_item < -1 || hooks->move_wait_ns < 0 || hooks->move_wait_ns > 10000000000ll)
        return EP_ERR_INVALID_ARG;
    ctx->hooks = *hooks;
    return EP_OK;
}

}  // extern "C"
