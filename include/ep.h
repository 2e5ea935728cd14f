/*
 * ep.h — C ABI of libep.so: MoE dispatch / combine for one GB300 (sm_103a).
 *
 * The operations are the expert-parallel (EP) exchange of DeepEP as described
 * by "如何突破MoE通信瓶颈：DeepEP跨节点优化技术终极指南" (cyqw.cn):
 *   - section 核心API示例: low_latency_dispatch(hidden_states, topk_idx,
 *     num_max_dispatch_tokens_per_rank, num_experts) and
 *     low_latency_combine(hidden_states, topk_idx, topk_weights, handle,
 *     num_experts);
 *   - section 技术解析: the dispatch layout is computed once and reused
 *     through a handle;
 *   - section 核心优势: FP8 dispatch and BF16 combine (128 tokens, hidden 7168,
 *     top-8 in the low-latency setting);
 *   - section 低延迟模式关键特性 / 性能调优: preallocated fixed-size receive
 *     buffers and a size hint (Buffer.get_low_latency_rdma_size_hint()).
 * The DeepTech announcement of DeepEP (010bt.com) adds the two kernel
 * families (low-latency and high-throughput "normal"), native FP8 dispatch
 * and SM-count control.
 *
 * Model.  R expert-parallel ranks are R *virtual* ranks whose send and receive
 * partitions all live in this GPU's memory.  Rank r holds T tokens
 * (T <= Tmax = num_max_dispatch_tokens_per_rank); token t of rank r is global
 * token g = r*T + t.  There are E experts (E % R == 0); expert e lives on rank
 * e / (E/R).  Each token picks K experts: topk_idx[g*K + k], -1 = none.
 *
 * Receive layout.  Every entry (g, k) with topk_idx != -1 gets one receive
 * row.  The rows of expert e start at base[e] and hold its entries in
 * ascending (g, k) order — deterministic, identical on every call.
 *   EP_LAYOUT_PADDED  (low-latency mode): E fixed buffers of R*Tmax rows,
 *                     base[e] = e*R*Tmax, rows = E*R*Tmax.  Rows past an
 *                     expert's count are never written.
 *   EP_LAYOUT_PACKED  (normal mode): base[e] = sum of the counts of experts
 *                     e' < e, rows = R*Tmax*K (worst case); rows past the
 *                     total count are never written.
 * Payload: BF16 rows [rows, H], or FP8 rows [rows, H] of OCP E4M3FN codes
 * plus fp32 scales [rows, H/128] (row-major).  FP8 cast per 128 channels of
 * a token: amax = max |x|, a = max(amax, 1e-4), scale = a/448 and
 * q = e4m3(x * (448/a)) rounded to nearest-even with saturation at +-448,
 * each step one IEEE fp32 operation.
 * Combine: out[g, c] = bf16( fma chain over k = 0..K-1 ascending of
 * w[g,k] * y[row(g,k), c], starting from +0, masked entries skipped ),
 * accumulated in fp32 and rounded once to bf16 (nearest-even).
 *
 * Conventions.
 *   - Pointers named d_* / documented "device" are device memory of the
 *     context's GPU; the caller allocates and owns them.  Everything else is
 *     host memory.
 *   - `stream` is a cudaStream_t (NULL = legacy default stream).  Calls only
 *     enqueue work: none of them synchronises the host, except
 *     ep_get_device_status and ep_autotune (which times candidates).
 *   - Errors a host can see (bad sizes, NULL pointers, misalignment) return at
 *     once and enqueue nothing.  Errors only the GPU can see (an expert id
 *     outside [-1, E), a padded expert buffer offered more than R*Tmax
 *     entries, a copy kernel's bounded wait giving up) set bits in a per-context
 *     device status word, read and cleared by ep_get_device_status; the
 *     offending entries get no row.
 *   - A context and its handles belong to the device current at ep_create;
 *     calls must be made with that device current.  A context is not
 *     thread-safe; calls on one context must not overlap on the GPU unless
 *     they use different handles and output buffers.
 */
#ifndef EP_H
#define EP_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define EP_ABI_VERSION 2

typedef enum ep_status {
    EP_OK = 0,
    EP_ERR_INVALID_ARG = 1,  /* a host-checkable argument is wrong; nothing enqueued */
    EP_ERR_UNSUPPORTED = 2,  /* valid but beyond the library's limits (see ep_config) */
    EP_ERR_OOM = 3,          /* a device allocation in ep_create / ep_handle_create failed */
    EP_ERR_CUDA = 4,         /* a CUDA runtime call or kernel launch failed */
    EP_ERR_BAD_EXPERT = 5,   /* device: a topk_idx entry was outside [-1, E) */
    EP_ERR_CAPACITY = 6,     /* device: padded layout, an expert was offered more than R*Tmax entries */
    EP_ERR_NO_LAYOUT = 7,    /* the handle holds no layout yet, or one for other sizes */
    EP_ERR_TIMEOUT = 8,      /* device: a bounded wait of a copy kernel gave up (about 1 s) */
    EP_ERR_TIMEOUT_IN_FLIGHT = 9  /* device: as EP_ERR_TIMEOUT, and the kernel's wait for its own
                                     row loads gave up too: a bulk load may have landed in shared
                                     memory after the kernel exited, so nothing the device ran
                                     afterwards can be trusted (start a new process) */
} ep_status;

typedef enum ep_layout {
    EP_LAYOUT_PADDED = 0,    /* low-latency mode: fixed-size per-expert buffers */
    EP_LAYOUT_PACKED = 1     /* normal mode: experts back to back (prefix sums) */
} ep_layout;

/* Sizes of one expert-parallel group.  Limits of the library:
 *   1 <= num_ranks <= 1024, 1 <= max_tokens_per_rank, 1 <= topk <= 32,
 *   num_experts % num_ranks == 0, 1 <= num_experts <= 1024,
 *   num_experts * num_ranks <= 16384,
 *   8 <= hidden <= 65536, hidden % 8 == 0 (FP8 dispatch: hidden % 128 == 0),
 *   receive rows and R*Tmax*K below 2^31, and a layout of fewer than
 *   (SM count) * 2^20 entries R*T*K (about 1.6e8 on 152 SMs; larger calls
 *   return EP_ERR_UNSUPPORTED).
 * max_sms caps the SMs the dispatch and combine kernels spread over (0 = all),
 * the SM-count control of the normal kernels. */
typedef struct ep_config {
    int32_t num_ranks;            /* R */
    int32_t max_tokens_per_rank;  /* Tmax (num_max_dispatch_tokens_per_rank) */
    int32_t hidden;               /* H, channels per token */
    int32_t num_experts;          /* E */
    int32_t topk;                 /* K */
    int32_t layout;               /* ep_layout */
    int32_t max_sms;              /* 0 = every SM */
} ep_config;

typedef struct ep_ctx ep_ctx;       /* a configured group + its device status word */
typedef struct ep_handle ep_handle; /* a cached dispatch layout (device buffers) */

/* Device buffers of a handle, for callers that consume the layout directly
 * (e.g. an expert kernel that needs src_info).  All pointers are device
 * pointers owned by the handle; contents are valid in stream order after the
 * ep_get_dispatch_layout / ep_dispatch call that filled them. */
typedef struct ep_handle_info {
    int32_t tokens_per_rank;   /* T of the layout held, -1 if none */
    int32_t num_tokens;        /* N = R*T */
    int64_t rows;              /* receive rows (ep_recv_rows) */
    int32_t *slot;             /* [N, K]  receive row of entry (g,k), -1 if none */
    int32_t *src_info;         /* [rows]  g*K + k of the entry in each written row */
    int32_t *cnt_er;           /* [E, R]  entries of source rank r for expert e */
    int32_t *off_er;           /* [E, R]  first row of (e, r) relative to base[e] */
    int64_t *base;             /* [E]     first receive row of expert e */
    int32_t *tokens_per_expert;/* [E]     rows expert e receives */
    int32_t has_rank_ranges;   /* 1: cnt_er / off_er belong to the layout held
                                  (ep_get_dispatch_layout computes them; the
                                  layout computed inside ep_dispatch does not) */
    int32_t rank_mode;         /* 1: a rank-deduplicated layout (ep_get_rank_layout):
                                  slot / src_info / base / tokens_per_expert are
                                  per destination rank ([R] instead of [E]) */
} ep_handle_info;

/* Human-readable name of a status code (static string). */
const char *ep_status_str(int32_t status);

/* EP_OK if cfg is within the limits above, else INVALID_ARG / UNSUPPORTED.
 * Touches no GPU. */
ep_status ep_config_check(const ep_config *cfg);

/* Receive rows of the configured layout (E*R*Tmax padded, R*Tmax*K packed).
 * Touches no GPU. */
ep_status ep_recv_rows(const ep_config *cfg, int64_t *rows);

/* Bytes the caller must allocate for the receive buffers, the analogue of
 * Buffer.get_low_latency_rdma_size_hint(): payload = rows*H*2 (BF16) or
 * rows*H (FP8); scales = rows*(H/128)*4 for FP8, else 0.  Touches no GPU. */
ep_status ep_recv_bytes(const ep_config *cfg, int32_t use_fp8,
                        uint64_t *payload_bytes, uint64_t *scale_bytes);

/* Create a context on the current device: validates cfg, allocates the
 * 4-byte device status word and reads the device's SM count.  *out is NULL on
 * error. */
ep_status ep_create(const ep_config *cfg, ep_ctx **out);
ep_status ep_destroy(ep_ctx *ctx);

/* Allocate a handle's device buffers (slot [R*Tmax*K], src_info [rows],
 * cnt_er/off_er [E*R], base/tokens_per_expert [E]) once, so that the calls
 * below allocate nothing and can be captured in a CUDA graph. */
ep_status ep_handle_create(ep_ctx *ctx, ep_handle **out);
ep_status ep_handle_destroy(ep_handle *handle);
ep_status ep_handle_get_info(const ep_handle *handle, ep_handle_info *out);

/* Dispatch layout (the "layout information" DeepEP computes once and reuses).
 *   d_topk_idx            device int64 [R, T, K], read only
 *   tokens_per_rank       T, 0 <= T <= Tmax
 *   d_num_tokens_per_rank device int32 [R] or NULL: tokens with >= 1 entry on rank d
 *   d_num_tokens_per_expert device int32 [E] or NULL: rows expert e receives
 *   d_is_token_in_rank    device uint8 [R*T, R] or NULL: 1 if token g has an
 *                         entry on rank d, else 0
 *   handle                receives slot / src_info / counts / bases
 * One kernel: a thread-block cluster, or from 128K entries (rank layout:
 * 48K) a cooperative kernel over all SMs (ep_tuning.layout_form forces
 * either); no host synchronisation.  If a launch fails (EP_ERR_CUDA /
 * EP_ERR_UNSUPPORTED) the handle holds no layout afterwards (the calls that
 * need one return EP_ERR_NO_LAYOUT); host-side argument errors leave it as
 * it was. */
ep_status ep_get_dispatch_layout(ep_ctx *ctx, const int64_t *d_topk_idx,
                                 int32_t tokens_per_rank,
                                 int32_t *d_num_tokens_per_rank,
                                 int32_t *d_num_tokens_per_expert,
                                 uint8_t *d_is_token_in_rank,
                                 ep_handle *handle, void *stream);

/* Rank-deduplicated layout, the transport of DeepEP's normal (high-
 * throughput) kernels (DeepTech announcement, 010bt.com: tokens forwarded per
 * destination domain; group-limited gating keeps the ranks per token low):
 * every token is sent ONCE to each rank that owns at least one of its experts
 * instead of once per expert.  The entry (g, k) that carries token g to rank
 * d is the first k of the token whose expert lives on d; the rows of rank d
 * start at d*R*Tmax (padded) or at the prefix of the per-rank counts
 * (packed) and hold its tokens in ascending g.  The handle then serves
 * ep_dispatch (topk_idx NULL; receive buffer of ep_rank_recv_rows rows, and
 * d_recv_count [R] gets the rows per rank) and ep_combine (weights NULL: the
 * token's rank rows are summed in the order their first expert appears in
 * its top-k row, fp32, one bf16 rounding; the expert side is expected to
 * have applied the weights of its local experts).
 *   d_topk_idx             device int64 [R, T, K]
 *   d_topk_weights         device fp32 [R*T, K] or NULL (all ones)
 *   d_num_tokens_per_rank  device int32 [R] or NULL: rows each rank receives
 *   d_recv_topk_idx        device int32 [rows, K] or NULL: per received row,
 *                          the token's local expert ids on that rank (e - d*E/R)
 *                          or -1 for experts on other ranks
 *   d_recv_topk_weights    device fp32 [rows, K] or NULL (needs d_recv_topk_idx):
 *                          the matching weights, 0 for other ranks' experts
 * Rows that receive nothing are not written. */
ep_status ep_get_rank_layout(ep_ctx *ctx, const int64_t *d_topk_idx, const float *d_topk_weights,
                             int32_t tokens_per_rank, int32_t *d_num_tokens_per_rank,
                             int32_t *d_recv_topk_idx, float *d_recv_topk_weights,
                             ep_handle *handle, void *stream);

/* Receive rows of the rank-deduplicated layout: R*R*Tmax (padded, every rank
 * can receive every token) or R*Tmax*min(K, R) (packed).  Touches no GPU. */
ep_status ep_rank_recv_rows(const ep_config *cfg, int64_t *rows);

/* low_latency_dispatch: scatter every token row to the receive rows of its
 * top-k experts, BF16 (bit copy) or FP8 (cast once per token, stored K times).
 *   d_x            device bf16 [R*T, H] (16-byte aligned), read only
 *   d_topk_idx     device int64 [R, T, K]: the layout is computed into handle
 *                  first (layout kernel + dispatch kernel); NULL: reuse the
 *                  layout already in handle (dispatch kernel only), except
 *                  that with tokens_per_rank == 0 an empty layout is computed
 *   tokens_per_rank T (must match the handle when reusing)
 *   use_fp8        0 = BF16 payload, 1 = FP8 payload + scales
 *   d_recv_x       device [rows, H] bf16 or uint8 (16-byte aligned)
 *   d_recv_scales  device fp32 [rows, H/128] (16-byte aligned) when use_fp8, else ignored
 *   d_recv_count   device int32 [E] or NULL: rows each expert received
 * Rows that receive nothing are not written. */
ep_status ep_dispatch(ep_ctx *ctx, const void *d_x, const int64_t *d_topk_idx,
                      int32_t tokens_per_rank, int32_t use_fp8, ep_handle *handle,
                      void *d_recv_x, float *d_recv_scales, int32_t *d_recv_count,
                      void *stream);

/* low_latency_combine: for each token, the fp32 weighted sum over its top-k
 * entries (ascending k, fused multiply-add) of the expert outputs found in
 * the entries' receive rows, rounded once to bf16.
 *   d_y            device bf16 [rows, H] in the handle's receive layout
 *                  (16-byte aligned), read only; only rows that received an
 *                  entry are read
 *   d_topk_weights device fp32 [R*T, K], or NULL for all weights 1 (the
 *                  backward of dispatch)
 *   handle         a layout from ep_get_dispatch_layout / ep_dispatch
 *   d_out          device bf16 [R*T, H] (16-byte aligned) */
ep_status ep_combine(ep_ctx *ctx, const void *d_y, const float *d_topk_weights,
                     const ep_handle *handle, void *d_out, void *stream);

/* Token-range forms of ep_dispatch and ep_combine on the layout already in
 * handle (the layout reuse of "如何突破MoE通信瓶颈：DeepEP跨节点优化技术终极指南",
 * section 技术解析: computed once, then reused by every later call), for a
 * caller that pipelines a step over chunks of tokens.  Global tokens are
 * g = r*T + t; a range [token_begin, token_end) must satisfy
 * 0 <= token_begin <= token_end <= R*T of the layout (else
 * EP_ERR_INVALID_ARG; no layout: EP_ERR_NO_LAYOUT); an empty range enqueues
 * nothing.  d_x, d_topk_weights and d_out are the full [R*T, ...] arrays, as
 * for ep_dispatch / ep_combine.  ep_dispatch_range writes the receive rows of
 * the range's entries (and nothing else; no counts); ep_combine_range writes
 * rows [token_begin, token_end) of d_out.  Ranges that together cover every
 * token give results identical, bit for bit, to one ep_dispatch (topk_idx
 * NULL) or ep_combine call.  One kernel each. */
ep_status ep_dispatch_range(ep_ctx *ctx, const void *d_x, int32_t use_fp8, const ep_handle *handle,
                            int64_t token_begin, int64_t token_end, void *d_recv_x,
                            float *d_recv_scales, void *stream);
ep_status ep_combine_range(ep_ctx *ctx, const void *d_y, const float *d_topk_weights,
                           const ep_handle *handle, int64_t token_begin, int64_t token_end,
                           void *d_out, void *stream);

/* Identity expert, the stand-in for the expert computation between dispatch
 * and combine in a round trip (FP8 dispatch / BF16 combine, same page,
 * section 核心优势).  For every receive row that an entry of a token in
 * [token_begin, token_end) received, writes that row of d_y with the BF16
 * value the row holds:
 *   use_fp8 = 1:  y[row, c] = bf16(e4m3(q[row, c]) * scale[row, c / 128])
 *                 (exact fp32 product, nearest-even bf16)
 *   use_fp8 = 0:  y[row] = recv[row] (bit copy; nothing to do when
 *                 d_y == d_recv_x)
 *   d_recv_x, d_recv_scales  what ep_dispatch wrote (read only)
 *   d_y            device bf16 [rows, H] (16-byte aligned); other rows are
 *                  not written
 * Range rules as for ep_dispatch_range.  One kernel. */
ep_status ep_expert_identity(ep_ctx *ctx, const ep_handle *handle, int32_t use_fp8,
                             const void *d_recv_x, const float *d_recv_scales, void *d_y,
                             int64_t token_begin, int64_t token_end, void *stream);

/* Split dispatch and combine: the send half returns and a later "hook" call
 * finishes the receive (the hook-based communication-computation overlap of
 * "如何突破MoE通信瓶颈：DeepEP跨节点优化技术终极指南", section 技术解析,
 * 通信-计算重叠技术; the DeepTech announcement of DeepEP, 010bt.com, says the
 * same).  Here the receive hooks and the combine send are copy kernels whose
 * threads only issue cp.async.bulk copies (the bulk-copy unit moves the
 * rows), so they can run on num_sms SMs (<= 0: the context's limit) while
 * other work uses the rest; they still occupy those SMs.  For a receive that
 * occupies no SM at all see the rank transport (ep_rank_dispatch_recv,
 * EP_WIRE_HOST) below.  The results are identical, bit for bit, to
 * ep_dispatch / ep_combine; the price is that every row crosses HBM once more
 * (through a send buffer).
 *
 * ep_dispatch_send: the layout (when d_topk_idx is given, as in ep_dispatch),
 *   then each token cast once (FP8) into its row of the send buffer:
 *     d_send_x       device [R*T, H] e4m3 (FP8) or bf16, 16-byte aligned; for
 *                    BF16 it may be d_x itself (then only the layout runs)
 *     d_send_scales  device fp32 [R*T, H/128], 16-byte aligned (FP8)
 * ep_dispatch_recv (the hook): every sent row copied to its receive rows,
 *   receive buffers and d_recv_count as ep_dispatch writes them.
 * ep_combine_send: the expert output of every received row copied back to the
 *   token-major buffer d_send_y [R*T*K, H] bf16 (row g*K + k for entry
 *   (g, k); rows of masked entries are not written).
 * ep_combine_recv (the hook): ep_combine over d_send_y (row g*K + k instead of
 *   the receive row), into d_out [R*T, H].
 * FP8 needs H % 512 == 0 here (EP_ERR_UNSUPPORTED otherwise).  A copy kernel's
 * waits for its row loads are bounded; if one gives up, the kernel stops and
 * ep_get_device_status reports EP_ERR_TIMEOUT. */
ep_status ep_dispatch_send(ep_ctx *ctx, const void *d_x, const int64_t *d_topk_idx,
                           int32_t tokens_per_rank, int32_t use_fp8, ep_handle *handle,
                           void *d_send_x, float *d_send_scales, void *stream);
ep_status ep_dispatch_recv(ep_ctx *ctx, const ep_handle *handle, int32_t use_fp8,
                           const void *d_send_x, const float *d_send_scales, void *d_recv_x,
                           float *d_recv_scales, int32_t *d_recv_count, int32_t num_sms,
                           void *stream);
ep_status ep_combine_send(ep_ctx *ctx, const ep_handle *handle, const void *d_y, void *d_send_y,
                          int32_t num_sms, void *stream);
ep_status ep_combine_recv(ep_ctx *ctx, const ep_handle *handle, const void *d_send_y,
                          const float *d_topk_weights, void *d_out, void *stream);

/* Rank-deduplicated transport with a receive that runs no kernel (the hook-
 * based overlap of "如何突破MoE通信瓶颈：DeepEP跨节点优化技术终极指南", section
 * 技术解析, 通信-计算重叠技术: the receive occupies no SM, and the page's figure
 * of the flow shows the CPU and GPU cooperating on the layout; the DeepTech
 * announcement of DeepEP, 010bt.com: the normal kernels forward tokens per
 * destination domain).  Tokens travel as in ep_get_rank_layout (once per
 * destination rank), and everything source rank r sends to rank d is ONE
 * contiguous run on both sides: the send buffer is ordered by (source rank,
 * destination rank, token), and the rows rank d receives hold its tokens in
 * ascending g = r*T + t.  A receive is then R*R copies, one per non-empty
 * run, issued from the host; no kernel of this library runs.  R <= 32
 * (EP_ERR_UNSUPPORTED otherwise).  Two wires move the runs:
 *   EP_WIRE_DEVICE  one device-to-device cudaMemcpyAsync per run (and one
 *                   per run of FP8 scales), spread over two internal
 *                   streams forked from and joined back into `stream`.
 *                   Runs at HBM speed; note that the CUDA driver carries out
 *                   same-device copies with its own kernels on the SMs (on
 *                   GB300 such copies wait for SMs held by other kernels).
 *   EP_WIRE_HOST    through the caller's pinned host buffer h_stage on the
 *                   copy engines only (device -> host, then host -> device,
 *                   pipelined per source rank): occupies no SM, at the host
 *                   link's speed (about 200 GB/s each way on GB300), the
 *                   role the network plays on the pages.  h_stage holds
 *                   ep_rank_send_rows rows of payload (H*2 bytes BF16, H
 *                   FP8), followed (FP8 dispatch) by as many rows of H/32
 *                   scale bytes; it must come from cudaMallocHost /
 *                   cudaHostAlloc (EP_ERR_INVALID_ARG otherwise).
 * The host needs the run sizes to issue the copies: the first wire call
 * after a new layout waits (host synchronisation) for the end of the
 * ep_rank_dispatch_send that computed it; later calls on the same layout
 * wait for nothing and only enqueue.
 *
 * ep_rank_send_rows: rows of a send buffer, R*Tmax*min(K, R).  Host only.
 * ep_rank_dispatch_send: the rank layout (as ep_get_rank_layout, outputs
 *   d_recv_topk_idx / d_recv_topk_weights optional) plus its run sizes and
 *   send rows, then each token cast once (FP8) and written to its send row
 *   for every destination rank; d_topk_idx NULL reuses the handle's layout
 *   (one made by this call, same tokens_per_rank: EP_ERR_NO_LAYOUT
 *   otherwise) and only casts.  Kernels: layout, send rows, dispatch.
 *     d_send_x       device [ep_rank_send_rows, H] e4m3 (FP8) or bf16
 *     d_send_scales  device fp32 [ep_rank_send_rows, H/128] (FP8)
 * ep_rank_dispatch_recv: the wire, send rows -> receive rows (and scales),
 *   receive buffers as ep_dispatch writes them for a rank layout
 *   (ep_rank_recv_rows rows), d_recv_count [R] the rows per rank.
 * ep_rank_combine_send: the wire back: the expert output of each received
 *   row (d_y, receive layout, bf16) to its send row of d_send_y
 *   [ep_rank_send_rows, H] bf16.
 * ep_rank_combine_recv: the rank-mode reduce (as ep_combine with weights
 *   NULL on a rank layout) reading each token's rows from d_send_y, into
 *   d_out [R*T, H].  One kernel.
 * ep_rank_runs: the run table (host arrays of R*R entries, [r*R + d]; any
 *   may be NULL): tokens source r sends to rank d, and the first send and
 *   receive row of each run.  May wait like the wire calls.
 * Results are identical, bit for bit, to ep_get_rank_layout + ep_dispatch /
 * ep_combine on the same routing. */
typedef enum ep_wire {
    EP_WIRE_DEVICE = 0,
    EP_WIRE_HOST = 1
} ep_wire;
ep_status ep_rank_send_rows(const ep_config *cfg, int64_t *rows);
ep_status ep_rank_dispatch_send(ep_ctx *ctx, const void *d_x, const int64_t *d_topk_idx,
                                const float *d_topk_weights, int32_t tokens_per_rank, int32_t use_fp8,
                                int32_t *d_recv_topk_idx, float *d_recv_topk_weights, ep_handle *handle,
                                void *d_send_x, float *d_send_scales, void *stream);
ep_status ep_rank_dispatch_recv(ep_ctx *ctx, ep_handle *handle, int32_t use_fp8, const void *d_send_x,
                                const float *d_send_scales, void *d_recv_x, float *d_recv_scales,
                                int32_t *d_recv_count, int32_t wire, void *h_stage, void *stream);
ep_status ep_rank_combine_send(ep_ctx *ctx, ep_handle *handle, const void *d_y, void *d_send_y,
                               int32_t wire, void *h_stage, void *stream);
ep_status ep_rank_combine_recv(ep_ctx *ctx, const ep_handle *handle, const void *d_send_y, void *d_out,
                               void *stream);
ep_status ep_rank_runs(ep_handle *handle, int32_t *run_cnt, int64_t *send_off, int64_t *recv_off);

/* chunk_tokens of ep_round_trip that asks for the automatic chunk size. */
#define EP_CHUNK_AUTO (-1)

/* One dispatch -> identity expert -> combine round trip, pipelined over
 * chunks of chunk_tokens global tokens: the layout (when d_topk_idx is
 * given, as in ep_dispatch), then for each chunk ep_dispatch_range,
 * ep_expert_identity and ep_combine_range, each kernel started early behind
 * the one before it (programmatic dependent launch).  A chunk's receive
 * rows are read back soon after they are written, while they can still be
 * in L2.  chunk_tokens: 0 (or >= R*T) is one chunk, EP_CHUNK_AUTO the size
 * ep_round_trip_auto_chunk gives, below -1 EP_ERR_INVALID_ARG.  d_out is
 * identical, bit for bit, for every chunk size.  Arguments as for the calls
 * it makes; d_y may equal d_recv_x for BF16. */
ep_status ep_round_trip(ep_ctx *ctx, const void *d_x, const int64_t *d_topk_idx,
                        int32_t tokens_per_rank, const float *d_topk_weights, int32_t use_fp8,
                        ep_handle *handle, void *d_recv_x, float *d_recv_scales, void *d_y,
                        void *d_out, int32_t chunk_tokens, void *stream);

/* The chunk size EP_CHUNK_AUTO stands for: the most tokens whose receive
 * rows (payload, FP8 scales and the bf16 expert output: K rows per token,
 * min(K, R) for a rank-deduplicated layout when rank_layout != 0) take
 * about 70% of the device's L2, rounded down to a multiple of 64 tokens, at
 * least 64 — or the tuned size when ep_set_tuning / ep_autotune set one.
 * Host only. */
ep_status ep_round_trip_auto_chunk(const ep_ctx *ctx, int32_t use_fp8, int32_t rank_layout,
                                   int32_t *chunk_tokens);

/* Launch shapes of a context ("run all tests and use the best auto-tuned
 * setting", DeepTech announcement of DeepEP, 010bt.com; SM control of
 * "如何突破MoE通信瓶颈：DeepEP跨节点优化技术终极指南", section 功能4).  None of
 * them changes a result bit: they only decide how the work is spread.
 *   dispatch_ctas_per_sm  CTAs per SM of the row dispatch kernel (1..16),
 *                         0 = the built-in rule (from H; at most 4 for FP8)
 *   combine_chunks        256-channel chunks per combine work item (1, 2 or 4),
 *                         0 = the built-in rule (from the entries per token)
 *   round_trip_chunk      tokens per chunk that EP_CHUNK_AUTO stands for in
 *                         ep_round_trip; 0 = the L2 rule; >= R*T (INT32_MAX
 *                         from ep_autotune) = one chunk
 *   dispatch_kernel       0 = the built-in rule (the warp-item kernel for FP8
 *                         rows of H <= 1024, or H <= 2048 with topk <= 4; else
 *                         the token kernel from 64K receive rows (tokens x
 *                         topk) on all SMs; else the row kernel where it
 *                         applies), 1 = the row kernel (bulk copies of whole
 *                         rows; only where H % 512 == 0 and H <= 15872, the
 *                         warp-item kernel elsewhere), 2 = the warp-item kernel
 *                         (16-byte stores by every lane), 3 = the token kernel
 *                         (one CTA per token holding its row in registers,
 *                         16-byte stores of the whole row per entry; where
 *                         H % 16 == 0 (FP8: H % 128 == 0) and H <= 16384, the
 *                         rule's kernel elsewhere)
 *   layout_form           0 = the built-in rule (one thread-block cluster below
 *                         a size, the grid form over all SMs from it), 1 = the
 *                         cluster, 2 = the grid form (one cooperative kernel;
 *                         the cluster where it cannot run) */
typedef struct ep_tuning {
    int32_t dispatch_ctas_per_sm;
    int32_t combine_chunks;
    int32_t round_trip_chunk;
    int32_t dispatch_kernel;
    int32_t layout_form;
} ep_tuning;

/* One candidate ep_autotune timed: knob (EP_TUNE_*), its value, median µs. */
typedef enum ep_tune_knob {
    EP_TUNE_DISPATCH = 0,              /* value 100 * dispatch_kernel + dispatch_ctas_per_sm;
                                          timed as layout + dispatch */
    EP_TUNE_COMBINE_CHUNKS = 1,
    EP_TUNE_ROUND_TRIP_CHUNK = 2,      /* INT32_MAX: one chunk */
    EP_TUNE_LAYOUT_FORM = 3            /* timed as layout + dispatch */
} ep_tune_knob;
typedef struct ep_tune_record {
    int32_t knob;
    int32_t value;
    float median_us;
} ep_tune_record;

ep_status ep_get_tuning(const ep_ctx *ctx, ep_tuning *out);
/* Values out of range: EP_ERR_INVALID_ARG and the tuning is unchanged. */
ep_status ep_set_tuning(ep_ctx *ctx, const ep_tuning *tuning);

/* Time each launch shape above on the caller's own inputs and keep the
 * fastest in the context (also written to *out; the built-in rule's choice is
 * timed first and kept unless another candidate is at least 3% faster):
 * layout + dispatch with the rule's layout form, the cluster and the grid
 * form, then with the rule's kernel, the row kernel at 1..4 CTAs per
 * SM (H % 512 == 0, H <= 15872) and the warp-item kernel, the combine with
 * 1, 2 and 4 chunks per item,
 * then the round trip in one chunk and in chunks of half, one and two times
 * the L2 rule.  Each candidate: the median of `reps` (1..1000) runs, before
 * each a write of twice the L2 size and a read of another twice the L2 size
 * (as behind kernels that just wrote a lot).  Arguments as for ep_round_trip
 * (d_topk_idx required, tokens_per_rank >= 1; d_y == d_recv_x tunes the BF16
 * round trip in place); d_recv_x / d_recv_scales / d_y / d_out are
 * overwritten.  Unlike the other calls it allocates (a handle and a 4x-L2
 * buffer, freed before it returns) and synchronises `stream`; on error the
 * previous tuning is kept. */
ep_status ep_autotune(ep_ctx *ctx, const void *d_x, const int64_t *d_topk_idx,
                      int32_t tokens_per_rank, const float *d_topk_weights, int32_t use_fp8,
                      void *d_recv_x, float *d_recv_scales, void *d_y, void *d_out, int32_t reps,
                      ep_tuning *out, void *stream);

/* The candidates the last ep_autotune on this context timed, in order (at
 * most 24): *count gets their number, records[0 .. min(count, capacity))
 * their values.  Host only. */
ep_status ep_get_autotune_log(const ep_ctx *ctx, ep_tune_record *records, int32_t capacity,
                              int32_t *count);

/* Dispatch for callers that cannot allocate device memory (no counterpart on
 * the pages: it is this library's own addition).  Same operation and output as
 * ep_dispatch with d_topk_idx given (layout, then BF16 copy or FP8 cast into
 * d_recv_x / d_recv_scales, rows per expert into d_recv_count), but it needs
 * no context or handle: every intermediate buffer lives in one static device
 * array that libep.so holds on each GPU that loads it (about 4.3 MB, kept
 * until the process exits).  It calls no cudaMalloc, cudaFree or allocating
 * library routine, so runtimes that give all device memory to their own
 * allocator up front, plugins that may only use the memory they are handed,
 * and latency-critical code where a cudaMalloc could synchronise the device
 * can still dispatch.
 *   cfg            sizes and layout, as for ep_create (host pointer)
 *   other args     as for ep_dispatch
 * Limits: R*tokens_per_rank*K <= 65536 entries, receive rows <= 1048576,
 * num_experts <= 1024; beyond them it returns EP_ERR_UNSUPPORTED and enqueues
 * nothing (a launch the device refuses returns EP_ERR_UNSUPPORTED too, after
 * the clear of the array's status word has been enqueued).  The first call on
 * a device looks up the array's device address (cudaGetSymbolAddress) and sets
 * kernel attributes; make it before any stream capture.  Every call looks the
 * address up again and repeats that set-up if it moved (a cudaDeviceReset
 * loads the module anew).  All calls share the array and each clears the
 * status word it uses first: calls whose work overlaps on the GPU race.
 * Device-detected errors (ids outside [-1, E), padded overflow) drop the
 * offending entries as in ep_dispatch but are not reported (there is no
 * context to report them to). */
ep_status ep_dispatch_noalloc(const ep_config *cfg, const void *d_x, const int64_t *d_topk_idx,
                              int32_t tokens_per_rank, int32_t use_fp8, void *d_recv_x,
                              float *d_recv_scales, int32_t *d_recv_count, void *stream);

/* Synchronise `stream`, read and clear the context's device status word.
 * Returns EP_OK, EP_ERR_BAD_EXPERT, EP_ERR_CAPACITY, EP_ERR_TIMEOUT_IN_FLIGHT,
 * EP_ERR_TIMEOUT or EP_ERR_CUDA (the first that applies, in this order). */
ep_status ep_get_device_status(ep_ctx *ctx, void *stream);

/* Test-only switches of a context (this library's own addition; the pages
 * have no counterpart), for running a failure path that real inputs never
 * reach without faulting or hanging the GPU:
 *   move_withhold_item  an item of the copy kernels of ep_dispatch_recv (token
 *                       g) and ep_combine_send (entry g*K + k) whose row load
 *                       is never issued, so the bounded wait for it runs out
 *                       and ep_get_device_status reports EP_ERR_TIMEOUT (no
 *                       load is in flight for it); -1 = none (the default)
 *   move_wait_ns        bound of each of those waits in ns; 0 = 1 s (the
 *                       default), at most 10 s
 * Values out of range: EP_ERR_INVALID_ARG and the switches are unchanged.
 * Host only. */
typedef struct ep_test_hooks {
    int64_t move_withhold_item;
    int64_t move_wait_ns;
} ep_test_hooks;
ep_status ep_set_test_hooks(ep_ctx *ctx, const ep_test_hooks *hooks);

#ifdef __cplusplus
}
#endif

#endif /* EP_H */
