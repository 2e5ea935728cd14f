/* The C ABI of libep.so used from plain C11, with no Python in between: the
 * header compiles as C, the library links, and the calls that need no GPU
 * (limits, sizes, status names, host-side argument checks) answer as the
 * header documents.  Prints "ok" and exits 0 when every check holds. */
#include <stdio.h>
#include <string.h>

#include "ep.h"

static int fails = 0;
#define CHECK(c)                                                          \
    do {                                                                  \
        if (!(c)) {                                                       \
            printf("FAIL %s:%d: %s\n", __FILE__, __LINE__, #c);           \
            fails++;                                                      \
        }                                                                 \
    } while (0)

int main(void) {
    /* the low-latency setting: 32 ranks x 128 tokens, H = 7168, 256 experts, top-8 */
    ep_config c = {32, 128, 7168, 256, 8, EP_LAYOUT_PADDED, 0};
    CHECK(ep_config_check(&c) == EP_OK);

    int64_t rows = 0;
    CHECK(ep_recv_rows(&c, &rows) == EP_OK);
    CHECK(rows == 256LL * 32 * 128);                 /* E * R * Tmax */
    uint64_t payload = 0, scales = 0;
    CHECK(ep_recv_bytes(&c, 1, &payload, &scales) == EP_OK);
    CHECK(payload == (uint64_t)rows * 7168);         /* e4m3 codes */
    CHECK(scales == (uint64_t)rows * (7168 / 128) * 4);
    CHECK(ep_recv_bytes(&c, 0, &payload, &scales) == EP_OK);
    CHECK(payload == (uint64_t)rows * 7168 * 2 && scales == 0);
    CHECK(ep_rank_recv_rows(&c, &rows) == EP_OK && rows == 32LL * 32 * 128);
    CHECK(ep_rank_send_rows(&c, &rows) == EP_OK && rows == 32LL * 128 * 8);  /* R*Tmax*min(K, R) */
    ep_test_hooks hooks = {-2, 0};
    CHECK(ep_set_test_hooks(NULL, &hooks) == EP_ERR_INVALID_ARG);

    ep_config packed = c;
    packed.layout = EP_LAYOUT_PACKED;
    CHECK(ep_recv_rows(&packed, &rows) == EP_OK && rows == 32LL * 128 * 8);
    CHECK(ep_rank_recv_rows(&packed, &rows) == EP_OK && rows == 32LL * 128 * 8);

    ep_config bad = c;
    bad.num_experts = 250;                           /* not a multiple of R */
    CHECK(ep_config_check(&bad) == EP_ERR_INVALID_ARG);
    bad = c;
    bad.topk = 33;                                   /* past the top-k limit */
    CHECK(ep_config_check(&bad) == EP_ERR_UNSUPPORTED);
    ep_config odd = c;
    odd.hidden = 200;                                /* FP8 needs H % 128 == 0 */
    CHECK(ep_recv_bytes(&odd, 1, &payload, &scales) == EP_ERR_UNSUPPORTED);
    CHECK(ep_config_check(NULL) == EP_ERR_INVALID_ARG);

    CHECK(strcmp(ep_status_str(EP_OK), "ok") == 0);
    CHECK(strcmp(ep_status_str(12345), "unknown status") == 0);

    /* host-side rejections happen before any device work */
    ep_ctx *ctx = (ep_ctx *)&c;
    CHECK(ep_create(&bad, &ctx) == EP_ERR_UNSUPPORTED && ctx == NULL);
    CHECK(ep_create(&c, NULL) == EP_ERR_INVALID_ARG);
    CHECK(ep_destroy(NULL) == EP_ERR_INVALID_ARG);
    CHECK(ep_handle_destroy(NULL) == EP_ERR_INVALID_ARG);
    CHECK(ep_get_dispatch_layout(NULL, NULL, 0, NULL, NULL, NULL, NULL, NULL) == EP_ERR_INVALID_ARG);
    CHECK(ep_dispatch(NULL, NULL, NULL, 0, 0, NULL, NULL, NULL, NULL, NULL) == EP_ERR_INVALID_ARG);
    CHECK(ep_combine(NULL, NULL, NULL, NULL, NULL, NULL) == EP_ERR_INVALID_ARG);
    CHECK(ep_dispatch_noalloc(&bad, NULL, NULL, 0, 0, NULL, NULL, NULL, NULL) == EP_ERR_UNSUPPORTED);
    int32_t chunk = 0;
    CHECK(ep_round_trip_auto_chunk(NULL, 1, 0, &chunk) == EP_ERR_INVALID_ARG);
    ep_tuning t;
    memset(&t, 0, sizeof t);
    CHECK(ep_get_tuning(NULL, &t) == EP_ERR_INVALID_ARG);

    printf("%s\n", fails ? "FAILED" : "ok");
    return fails != 0;
}
