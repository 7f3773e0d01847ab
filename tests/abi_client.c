/*
 * abi_client.c -- a plain C11 user of the library's C ABI (include/kivi.h):
 * compiled with gcc against the public header only (no CUDA headers) and
 * linked to libkivi_gb300.so. It calls the host-side entry points and the
 * argument checks that return before any launch, so it needs no GPU, and
 * prints one "name value" line per check for tests/test_c_client.py.
 *
 * Worked flush counts: VeloxQuant-MLX blog, "A 5.65x Metal Kernel That Made
 * My LLM Exactly 0% Faster", "The full end-to-end record" (559 -> 512,
 * 2059 -> 2016, 8209 -> 8160 at residual_length = group_size = 32).
 */
#include <stddef.h>
#include <stdio.h>

#include "kivi.h"

int main(void)
{
    printf("version %d\n", kivi_version());
    printf("status_ok %s\n", kivi_status_string(KIVI_OK));
    printf("status_unsupported %s\n", kivi_status_string(KIVI_ERR_UNSUPPORTED));
    printf("flush_559 %d\n", kivi_flush_count(559, 32, 32));
    printf("flush_2059 %d\n", kivi_flush_count(2059, 32, 32));
    printf("flush_8209 %d\n", kivi_flush_count(8209, 32, 32));
    printf("flush_all_ragged %d\n", kivi_flush_count(77, 0, 32));
    printf("flush_bad %d\n", kivi_flush_count(-1, 32, 32));

    /* checks that fail before any launch: no device memory is touched */
    int n = -7;
    printf("flush_bad_bits %d\n", (int)kivi_flush_keys(NULL, 8, 256, 256, 128, 32, 3, 128,
                                                      NULL, NULL, NULL, 0, 256, &n, NULL));
    printf("flush_bad_dim %d\n", (int)kivi_flush_values(NULL, 8, 256, 256, 96, 32, 4, 128,
                                                       NULL, NULL, NULL, 0, 256, &n, NULL));
    printf("flush_null_x %d\n", (int)kivi_flush_keys(NULL, 8, 256, 256, 128, 32, 4 | KIVI_SCALE_F16, 128,
                                                    NULL, NULL, NULL, 0, 256, &n, NULL));
    n = -7;
    kivi_status st = kivi_flush_keys(NULL, 8, 100, 100, 128, 32, 4, 128, NULL, NULL, NULL, 0, 256, &n, NULL);
    printf("flush_nothing %d %d\n", (int)st, n); /* nothing to flush: OK, no pointer needed */
    printf("dequant_empty %d\n", (int)kivi_dequant(KIVI_AXIS_VALUES, NULL, NULL, NULL, 8, 0, 128, 32, 4,
                                                   256, NULL, NULL));
    printf("residual_bad_dim %d\n", (int)kivi_residual_append(NULL, 4, 4, NULL, 8, 160, 96, 0, NULL));

    size_t ws = kivi_decode_workspace_size(1, 32, 8, 2080, 158, 128);
    printf("workspace_qwen8b_positive %d\n", ws > KIVI_DECODE_COUNTER_BYTES ? 1 : 0);
    printf("workspace_one_tile %zu\n", kivi_decode_workspace_size(1, 32, 8, 32, 0, 128));
    printf("decode_no_workspace %d\n",
           (int)kivi_decode_attend((const void*)16, (const void*)16, (const float*)16, (const void*)16,
                                   (const void*)16, (const float*)16, (const void*)16, 2080, 2080,
                                   (const void*)16, (const void*)16, 158, 160, 1, 32, 8, 128, 32, 4,
                                   0.088f, (float*)16, NULL, 0, NULL));
    printf("decode_bad_group %d\n",
           (int)kivi_decode_attend(NULL, NULL, NULL, NULL, NULL, NULL, NULL, 2080, 2080, NULL, NULL, 158,
                                   160, 1, 32, 8, 128, 32, 4, 0.088f, NULL, NULL, 0, NULL) );
    printf("decode_too_many_heads %d\n",
           (int)kivi_decode_attend(NULL, NULL, NULL, NULL, NULL, NULL, NULL, 2080, 2080, NULL, NULL, 158,
                                   160, 1, 8 * 65, 8, 128, 32, 4, 0.088f, NULL, NULL, 0, NULL));
    printf("workspace_init_null %d\n", (int)kivi_decode_workspace_init(NULL, 1024, NULL));
    int info[7] = {0};
    st = kivi_decode_plan_info(1, 32, 8, 2080, 158, 128, 32, 4, info);
    printf("plan_qwen8b %d %d %d %d\n", (int)st, info[0], info[1], info[5]); /* status, pair kernel, splits, tiles */
    st = kivi_decode_plan_info(1, 32, 8, 2080, 158, 128, 32, 4 | KIVI_SCALE_F16, info);
    printf("plan_qwen8b_f16s %d %d\n", (int)st, info[0]);

    /* the layer cache: the struct's layout as C sees it, and its checks
       (never-dereferenced 16-byte aligned addresses) */
    printf("cache_layout %zu %zu %zu %zu %zu\n", sizeof(kivi_cache), offsetof(kivi_cache, kcodes),
           offsetof(kivi_cache, S_q), offsetof(kivi_cache, store_written), offsetof(kivi_cache, res_off));
    void* a = (void*)256;
    kivi_cache c = {8, 128, 32, 4, 128, 256, 160, a, (float*)a, a, a, (float*)a, a, a, a, 0, 0, 0, 0};
    n = -7;
    st = kivi_cache_prefill(&c, a, a, 0, 0, &n, NULL);
    printf("cache_prefill_nothing %d %d\n", (int)st, n);
    c.res_off = 100;
    c.n_res = 61;
    st = kivi_cache_append(&c, a, a, 1, 1, &n, NULL);
    printf("cache_window_past_end %d %d %d\n", (int)st, c.n_res, c.res_off);
    c.res_off = 0;
    c.n_res = 0;
    printf("cache_decode_bad_batch %d\n",
           (int)kivi_cache_decode(&c, a, 2, 32, 8, 0.088f, (float*)a, a, (size_t)1 << 30, NULL));
    return 0;
}
