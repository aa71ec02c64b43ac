/*
 * A plain C11 caller of the MLA decode library: the header compiles as C and
 * the shared library links and answers the calls that need no GPU (status
 * strings, workspace sizes, argument checks that fail before any launch).
 * Built and run by tests/test_abi.py; prints "ok" and exits 0 on success.
 */
#include <stdio.h>
#include <string.h>

#include "mla_decode.h"

#define CHECK(cond)                                                         \
    do {                                                                    \
        if (!(cond)) {                                                      \
            fprintf(stderr, "failed: %s (line %d)\n", #cond, __LINE__);     \
            return 1;                                                       \
        }                                                                   \
    } while (0)

int main(void) {
    CHECK(strcmp(mla_status_string(MLA_OK), "ok") == 0);
    CHECK(strcmp(mla_status_string(MLA_ERR_WORKSPACE), "workspace too small") == 0);
    CHECK(mla_workspace_bytes(64, 1, 128, 1, MLA_V_DIM, 76) > 0);
    CHECK(mla_workspace_bytes(64, 1, 128, 1, 256, 76) == 0);
    CHECK(MLA_FP8_PAGE_BYTES(MLA_HEAD_DIM) == 37120);
    int parts = 0;
    CHECK(mla_num_sm_parts(0, 128, 1, NULL) == MLA_ERR_INVALID_ARG);
    CHECK(mla_num_sm_parts(0, 128, 2, &parts) == MLA_ERR_UNSUPPORTED);
    CHECK(mla_get_metadata(NULL, 2, 16, 1, 3, NULL, NULL, NULL) == MLA_ERR_INVALID_ARG);
    /* every decode entry rejects a missing query before touching the GPU */
    CHECK(mla_decode_kvcache(NULL, NULL, 1, NULL, 1, NULL, 1, 1, 16, 1, MLA_HEAD_DIM, MLA_V_DIM, NULL, NULL, 1,
                             0.04f, 0, NULL, NULL, NULL, 0, NULL) == MLA_ERR_INVALID_ARG);
    CHECK(mla_decode_kvcache_fp8(NULL, NULL, 1, NULL, 1, NULL, 1, 1, 16, 1, MLA_HEAD_DIM, MLA_V_DIM, NULL, NULL, 1,
                                 0.04f, 0, NULL, NULL, NULL, 0, NULL) == MLA_ERR_INVALID_ARG);
    CHECK(mla_decode_kvcache_sparse(NULL, NULL, 1, NULL, 1, NULL, NULL, 64, NULL, 1, 1, 16, 1, MLA_HEAD_DIM,
                                    MLA_V_DIM, NULL, NULL, 1, 0.04f, NULL, NULL, NULL, 0, NULL) == MLA_ERR_INVALID_ARG);
    CHECK(mla_decode_kvcache_noalloc(NULL, NULL, 1, NULL, 1, NULL, 1, 1, 16, 1, MLA_HEAD_DIM, MLA_V_DIM, NULL, NULL,
                                     1, 0.04f, 0, NULL, NULL, NULL) == MLA_ERR_INVALID_ARG);
    CHECK(mla_set_timing_events(NULL, (void *)1) == MLA_ERR_INVALID_ARG);
    printf("ok\n");
    return 0;
}
