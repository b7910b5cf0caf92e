/*
 * The C ABI used from plain C99: every entry point declared in pagedattn.h is
 * bound to a function pointer of the type written out here (a declaration that
 * drifted from it does not compile), and each is called in a way that returns
 * before any CUDA call: status names, empty batches, argument errors.
 */
#include <stdio.h>
#include <string.h>

#include "pagedattn.h"

int main(void)
{
    /* every entry point, through a pointer of its declared type */
    const char *(*status_name)(pa_status_t) = pa_status_string;
    pa_status_t (*store)(const void *, const void *, void *, void *, const int64_t *, int64_t,
                         int, int, int, int64_t, void *) = pa_store_kvcache;
    pa_status_t (*store_layout)(const void *, const void *, void *, void *, const int64_t *,
                                int64_t, int, int, int, int64_t, pa_layout_t, void *) =
        pa_store_kvcache_layout;
    size_t (*ws_size)(int, int, int, int) = pa_decode_workspace_size;
    pa_status_t (*decode)(const void *, const void *, const void *, const int32_t *, int,
                          const int32_t *, float, void *, int, int, int, int, int, int64_t,
                          void *, size_t, void *) = pa_decode;
    pa_status_t (*splitk)(const void *, const void *, const void *, const int32_t *, int,
                          const int32_t *, float, void *, int, int, int, int, int, int64_t,
                          void *, size_t, int, void *) = pa_decode_splitk;
    pa_status_t (*noalloc)(const void *, const void *, const void *, const int32_t *, int,
                           const int32_t *, float, void *, int, int, int, int, int, int64_t,
                           void *) = pa_decode_noalloc;
    pa_status_t (*decode_layout)(const void *, const void *, const void *, const int32_t *, int,
                                 const int32_t *, float, void *, int, int, int, int, int,
                                 int64_t, pa_layout_t, void *, size_t, int, void *) =
        pa_decode_layout;
    size_t (*multi_ws_size)(int, int, int, int) = pa_decode_multi_workspace_size;
    pa_status_t (*multi)(const void *, const void *, const void *, const int32_t *, int,
                         const int32_t *, int, float, void *, int, int, int, int, int, int64_t,
                         void *, size_t, void *) = pa_decode_multi;
    pa_status_t (*multi_layout)(const void *, const void *, const void *, const int32_t *, int,
                                const int32_t *, int, float, void *, int, int, int, int, int,
                                int64_t, pa_layout_t, void *, size_t, void *) =
        pa_decode_multi_layout;
    pa_status_t (*prefill)(const void *, const void *, const void *, const int32_t *, int,
                           const int32_t *, const int32_t *, int, float, void *, int, int, int,
                           int, int, int, int64_t, void *) = pa_prefill;
    pa_status_t (*prefill_layout)(const void *, const void *, const void *, const int32_t *,
                                  int, const int32_t *, const int32_t *, int, float, void *, int,
                                  int, int, int, int, int, int64_t, pa_layout_t, void *) =
        pa_prefill_layout;
    pa_status_t (*step)(const void *, const void *, const int64_t *, int64_t, const void *,
                        void *, void *, const int32_t *, int, const int32_t *, float, void *, int,
                        int, int, int, int, int64_t, pa_layout_t, void *, size_t, void *) =
        pa_decode_step;
    pa_status_t (*take_error)(int32_t *, void *) = pa_take_device_error;
    pa_status_t (*fault_hook)(int) = pa_debug_prefill_fault;
    pa_status_t (*variant_hook)(int) = pa_debug_kernel_variant;
    int failures = 0;

    if (strcmp(status_name(PA_ERR_WORKSPACE), "PA_ERR_WORKSPACE") != 0)
        ++failures;
    /* empty work: PA_OK without touching a device */
    if (store(NULL, NULL, NULL, NULL, NULL, 0, 8, 128, 16, 10, NULL) != PA_OK)
        ++failures;
    if (decode(NULL, NULL, NULL, NULL, 4, NULL, 0.1f, NULL, 0, 16, 8, 128, 16, 10, NULL, 0,
               NULL) != PA_OK)
        ++failures;
    if (prefill(NULL, NULL, NULL, NULL, 4, NULL, NULL, 8, 0.1f, NULL, 0, 0, 16, 8, 128, 16, 10,
                NULL) != PA_OK)
        ++failures;
    if (store_layout(NULL, NULL, NULL, NULL, NULL, 0, 8, 128, 16, 10, PA_LAYOUT_HEAD_MAJOR,
                     NULL) != PA_OK)
        ++failures;
    if (multi(NULL, NULL, NULL, NULL, 4, NULL, 2, 0.1f, NULL, 0, 16, 8, 128, 16, 10, NULL, 0,
              NULL) != PA_OK)
        ++failures;
    if (prefill_layout(NULL, NULL, NULL, NULL, 4, NULL, NULL, 8, 0.1f, NULL, 0, 0, 16, 8, 128,
                       16, 10, PA_LAYOUT_HEAD_MAJOR, NULL) != PA_OK)
        ++failures;
    /* argument errors are statuses (or a zero size) */
    if (take_error(NULL, NULL) != PA_ERR_INVALID_ARG)
        ++failures;
    if (fault_hook(5) != PA_ERR_INVALID_ARG)
        ++failures;
    if (ws_size(12, 8, 128, 0) != 0 || multi_ws_size(0, 16, 8, 128) != 0)
        ++failures;
    if (splitk(NULL, NULL, NULL, NULL, 4, NULL, 0.1f, NULL, 2, 16, 8, 128, 16, 10, NULL, 0, -1,
               NULL) != PA_ERR_INVALID_ARG)
        ++failures;
    if (noalloc(NULL, NULL, NULL, NULL, 4, NULL, 0.1f, NULL, 2, 16, 8, 64, 16, 10, NULL) !=
        PA_ERR_UNSUPPORTED)
        ++failures;
    /* pa_decode_noalloc answers like pa_decode: an empty batch is PA_OK with
     * no device (this program runs with none visible), bad head counts are
     * argument errors */
    if (noalloc(NULL, NULL, NULL, NULL, 4, NULL, 0.1f, NULL, 0, 16, 8, 128, 16, 10, NULL) != PA_OK)
        ++failures;
    if (noalloc(NULL, NULL, NULL, NULL, 4, NULL, 0.1f, NULL, 0, 64, 4, 128, 16, 10, NULL) != PA_OK)
        ++failures;
    if (noalloc(NULL, NULL, NULL, NULL, 4, NULL, 0.1f, NULL, 2, 12, 8, 128, 16, 10, NULL) !=
        PA_ERR_INVALID_ARG)
        ++failures;
    if (noalloc(NULL, NULL, NULL, NULL, 4, NULL, 0.1f, NULL, 2, 0, 8, 128, 16, 10, NULL) !=
        PA_ERR_INVALID_ARG)
        ++failures;
    if (noalloc(NULL, NULL, NULL, NULL, 4, NULL, 0.1f, NULL, 2, 16, 8, 128, 16, 10, NULL) !=
        PA_ERR_INVALID_ARG)
        ++failures;
    if (variant_hook(4) != PA_ERR_INVALID_ARG || variant_hook(0) != PA_OK)
        ++failures;
    /* a step with nothing to store and no sequence does nothing; a bad store
     * argument is reported before the decode's */
    if (step(NULL, NULL, NULL, 0, NULL, NULL, NULL, NULL, 4, NULL, 0.1f, NULL, 0, 16, 8, 128, 16,
             10, PA_LAYOUT_TOKEN_MAJOR, NULL, 0, NULL) != PA_OK)
        ++failures;
    if (step(NULL, NULL, NULL, 3, NULL, NULL, NULL, NULL, 4, NULL, 0.1f, NULL, 2, 16, 8, 128, 16,
             10, PA_LAYOUT_TOKEN_MAJOR, NULL, 0, NULL) != PA_ERR_INVALID_ARG)
        ++failures;
    if (step(NULL, NULL, NULL, 0, NULL, NULL, NULL, NULL, 4, NULL, 0.1f, NULL, 2, 16, 8, 64, 16,
             10, PA_LAYOUT_TOKEN_MAJOR, NULL, 0, NULL) != PA_ERR_UNSUPPORTED)
        ++failures;
    if (decode_layout(NULL, NULL, NULL, NULL, 4, NULL, 0.1f, NULL, 2, 16, 8, 128, 16, 10,
                      (pa_layout_t)3, NULL, 0, 0, NULL) != PA_ERR_INVALID_ARG)
        ++failures;
    if (multi_layout(NULL, NULL, NULL, NULL, 4, NULL, 17, 0.1f, NULL, 2, 16, 8, 128, 16, 10,
                     PA_LAYOUT_TOKEN_MAJOR, NULL, 0, NULL) != PA_ERR_UNSUPPORTED)
        ++failures;
    if (decode(NULL, NULL, NULL, NULL, 4, NULL, 0.1f, NULL, 2, 16, 8, 64, 16, 10, NULL, 0,
               NULL) != PA_ERR_UNSUPPORTED)
        ++failures;
    printf("%s %d\n", failures ? "FAIL" : "ok", failures);
    return failures ? 1 : 0;
}
