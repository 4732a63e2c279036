/* Plain C99 user of the library's public header: creates plans, reads the
 * sizes and status strings, and checks the documented rejections.  Touches
 * no GPU (plan calls are host only).  Prints "ok" and exits 0 on success. */
#include <stdio.h>
#include <string.h>

#include "tp.h"

#define CHECK(cond)                                                    \
    do {                                                               \
        if (!(cond)) {                                                 \
            fprintf(stderr, "%s:%d: check failed: %s\n", __FILE__, __LINE__, #cond); \
            return 1;                                                  \
        }                                                              \
    } while (0)

int main(void) {
    tp_plan_t plan = NULL;
    size_t packed = 0, ws = 0, ws_llama = 0;

    CHECK(tp_plan_create(4096, 32, 11008, 4, &plan) == TP_OK && plan != NULL);
    CHECK(tp_plan_sizes(plan, 1, 2048, &packed, &ws) == TP_OK);
    /* every weight once, bf16: 4 d^2 + 3 d f elements, plus section padding */
    CHECK(packed >= (size_t)2 * (4ull * 4096 * 4096 + 3ull * 4096 * 11008));
    CHECK(packed <= (size_t)2 * (4ull * 4096 * 4096 + 3ull * 4096 * 11008) + 4 * 1024);
    CHECK(ws > 0);
    tp_plan_destroy(plan);

    plan = (tp_plan_t)1;
    CHECK(tp_plan_create(4096, 32, 11008, 3, &plan) == TP_ERR_HEADS_NOT_DIVISIBLE && plan == NULL);
    CHECK(tp_plan_create(4096, 32, 11008, 64, &plan) == TP_ERR_DEGREE_RANGE);
    CHECK(tp_plan_create(4096, 32, 11001, 2, &plan) == TP_ERR_FFN_NOT_DIVISIBLE);
    CHECK(tp_plan_create_ex(256, 4, 1024, 2, TP_ACT_GELU, TP_FP32, &plan) == TP_OK);
    tp_plan_destroy(plan);

    CHECK(tp_plan_create_llama(4096, 32, 11008, 2, 1e-5f, 10000.0f, &plan) == TP_OK);
    CHECK(tp_plan_sizes(plan, 1, 2048, NULL, &ws_llama) == TP_OK && ws_llama > 0);
    CHECK(tp_column_linear(plan, TP_QKV, (const void*)0x10000, 4, (const void*)0x10000, (void*)0x10000, NULL, 0,
                           NULL) == TP_ERR_UNSUPPORTED);
    tp_plan_destroy(plan);

    CHECK(strcmp(tp_status_string(TP_OK), "TP_OK") == 0);
    CHECK(strcmp(tp_status_string(TP_ERR_DEVICE_TIMEOUT), "TP_ERR_DEVICE_TIMEOUT") == 0);
    CHECK(tp_last_cuda_error() != NULL);
    printf("ok\n");
    return 0;
}
