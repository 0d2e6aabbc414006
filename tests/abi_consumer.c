/* A plain C99 consumer of include/topk.h, linked against the built library.
 *
 * It shows that the header compiles as C (and, built a second time, as C++)
 * and that the documented host-side contract holds when called from C: the
 * workspace sizing, the status strings, and the status codes of calls that
 * fail validation. No call below reaches the GPU: each one either returns
 * before anything is enqueued or is an empty batch. The pointers are stand-ins
 * that the library never dereferences, because validation fails first.
 *
 * Prints "ok <n>" with the number of checks and exits 0, or prints the first
 * failed check and exits 1.
 */
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include "topk.h"

static int g_checks = 0;

#define CHECK(cond)                                                    \
    do {                                                               \
        ++g_checks;                                                    \
        if (!(cond)) {                                                 \
            printf("failed: %s (line %d)\n", #cond, __LINE__);         \
            return 1;                                                  \
        }                                                              \
    } while (0)

int main(void) {
    /* stand-ins: 16-byte aligned and not, never dereferenced */
    const float* scores = (const float*)(uintptr_t)0x10000u;
    const float* scores_unaligned = (const float*)(uintptr_t)0x10004u;
    const int32_t* ints = (const int32_t*)(uintptr_t)0x20000u;
    int32_t* out = (int32_t*)(uintptr_t)0x30000u;
    void* ws = (void*)(uintptr_t)0x40000u;
    const int32_t batch = 8;
    const size_t ws_bytes = topk_workspace_bytes(batch);
    int32_t rows = -1;
    uint32_t flags = 0;

    /* workspace sizing: a 256-byte multiple that grows with the batch */
    CHECK(topk_workspace_bytes(-1) == 0);
    CHECK(topk_workspace_bytes(0) > 0 && topk_workspace_bytes(0) % 256 == 0);
    CHECK(ws_bytes % 256 == 0 && ws_bytes >= topk_workspace_bytes(0));
    CHECK(topk_workspace_bytes(TOPK_NOALLOC_MAX_BATCH) >= topk_workspace_bytes(batch));

    /* status strings: one per code, and a fixed text for unknown codes */
    CHECK(strcmp(topk_status_string(TOPK_OK), topk_status_string(TOPK_ERR_K)) != 0);
    CHECK(topk_status_string(TOPK_ERR_CUDA) != NULL);
    CHECK(strcmp(topk_status_string(12345), "unknown status") == 0);

    /* plan: k outside [1, TOPK_MAX_K], a negative batch, a short workspace */
    CHECK(topk_plan(ints, batch, 0, ws, ws_bytes, NULL) == TOPK_ERR_K);
    CHECK(topk_plan(ints, batch, TOPK_MAX_K + 1, ws, ws_bytes, NULL) == TOPK_ERR_K);
    CHECK(topk_plan(ints, -1, 16, ws, ws_bytes, NULL) == TOPK_ERR_ARG);
    CHECK(topk_plan(ints, batch, 16, ws, ws_bytes - 1, NULL) == TOPK_ERR_WORKSPACE);

    /* PAGED: alignment of scores and stride, page size, flags */
    CHECK(topk_transform_paged(scores_unaligned, 64, NULL, ints, ints, 4, 64, batch, 16, ws, ws_bytes, out,
                               NULL, 0u, NULL) == TOPK_ERR_ALIGN);
    CHECK(topk_transform_paged(scores, 62, NULL, ints, ints, 4, 64, batch, 16, ws, ws_bytes, out, NULL, 0u,
                               NULL) == TOPK_ERR_ARG);
    CHECK(topk_transform_paged(scores, 64, NULL, ints, ints, 4, 48, batch, 16, ws, ws_bytes, out, NULL, 0u,
                               NULL) == TOPK_ERR_PAGE_SIZE);
    CHECK(topk_transform_paged(scores, 64, NULL, ints, ints, 4, TOPK_MAX_PAGE_SIZE * 2, batch, 16, ws, ws_bytes,
                               out, NULL, 0u, NULL) == TOPK_ERR_PAGE_SIZE);
    CHECK(topk_transform_paged(scores, 64, NULL, ints, ints, 4, 64, batch, 16, ws, ws_bytes, out, NULL,
                               TOPK_DETERMINISTIC << 1, NULL) == TOPK_ERR_ARG);

    /* packed PAGED: the page table is required, the workspace is checked */
    CHECK(topk_transform_paged_packed(scores, 64, NULL, ints, NULL, 4, 64, ints, ints, batch, 16, ws, ws_bytes,
                                      out, NULL, 0u, NULL) == TOPK_ERR_ARG);
    CHECK(topk_transform_paged_packed(scores, 64, NULL, ints, ints, 4, 64, ints, ints, batch, 16, NULL,
                                      ws_bytes, out, NULL, 0u, NULL) == TOPK_ERR_WORKSPACE);

    /* RAGGED: out_offsets is required; k is checked */
    CHECK(topk_transform_ragged(scores, 0, NULL, ints, NULL, batch, 16, ws, ws_bytes, out, NULL, 0u, NULL) ==
          TOPK_ERR_ARG);
    CHECK(topk_transform_ragged(scores, 0, NULL, ints, ints, batch, TOPK_MAX_K * 2, ws, ws_bytes, out, NULL,
                                0u, NULL) == TOPK_ERR_K);

    /* the built-in workspace has a batch limit, checked before any CUDA call */
    CHECK(topk_transform_ragged_noalloc(scores, 0, NULL, ints, ints, TOPK_NOALLOC_MAX_BATCH + 1, 16, out, NULL,
                                        0u, NULL) == TOPK_ERR_WORKSPACE);

    /* an empty batch is a no-op on every entry point */
    CHECK(topk_transform_ragged(NULL, 0, NULL, NULL, NULL, 0, 16, ws, topk_workspace_bytes(0), NULL, NULL, 0u,
                                NULL) == TOPK_OK);
    CHECK(topk_transform_paged(NULL, 0, NULL, NULL, NULL, 0, 1, 0, 16, ws, topk_workspace_bytes(0), NULL, NULL,
                               0u, NULL) == TOPK_OK);
    CHECK(topk_transform_ragged_noalloc(NULL, 0, NULL, NULL, NULL, 0, 16, NULL, NULL, 0u, NULL) == TOPK_OK);

    /* reading the device error words needs a workspace and the error-row output */
    CHECK(topk_read_device_errors(NULL, &rows, &flags, NULL) == TOPK_ERR_ARG);

    printf("ok %d\n", g_checks);
    return 0;
}
