/* A plain C consumer of libdsrows: it includes the public header, links the
 * shared library and makes calls that are answered on the host (sizes,
 * version, argument validation), so it runs without a GPU. Exit status 0
 * when every check holds; otherwise the failed check is printed. */
#include <stdio.h>
#include <string.h>

#include "dsrows.h"

static int failures = 0;

static void check(int ok, const char* what) {
    if (!ok) {
        fprintf(stderr, "FAILED: %s (last error: \"%s\")\n", what, ds_rows_last_error());
        ++failures;
    }
}

int main(void) {
    check(strstr(ds_rows_version(), "sm_103a") != NULL, "version names the target");

    /* Sizes: an empty table is invalid, a valid one needs a workspace. */
    check(ds_rows_workspace_bytes(0, NULL) == 0, "no rows: no workspace size");
    check(strlen(ds_rows_last_error()) > 0, "the rejection leaves a message");
    ds_row_t rows[2] = {{4096, 512, 0, 0}, {300, 300, 512, 1}};
    const size_t ws = ds_rows_workspace_bytes(2, rows);
    check(ws > 0 && ws % 256 == 0, "a valid table needs a 256-byte multiple");

    /* Validation: a bad call enqueues nothing and returns a DS_E* code. */
    const ds_bf16* keys[2] = {(const ds_bf16*)0x7f0000000000ull, (const ds_bf16*)0x7f0000010000ull};
    ds_row_set_t set = {9, rows, keys, keys};
    check(ds_rows_decode(&set, (const ds_bf16*)keys[0], (const float*)keys[0], (const ds_bf16*)keys[0],
                         (const float*)keys[0], 0, 0.044f, (ds_bf16*)keys[0], NULL, NULL, (void*)keys[0], ws,
                         NULL) == DS_EINVAL,
          "nine rows are rejected");
    set.rows = 2;
    check(ds_rows_decode(&set, (const ds_bf16*)keys[0], (const float*)keys[0], (const ds_bf16*)keys[0],
                         (const float*)keys[0], 0, -1.0f, (ds_bf16*)keys[0], NULL, NULL, (void*)keys[0], ws,
                         NULL) == DS_EINVAL,
          "a negative scale is rejected");
    check(ds_rows_decode(&set, (const ds_bf16*)keys[0], (const float*)keys[0], (const ds_bf16*)keys[0],
                         (const float*)keys[0], 0, 0.044f, (ds_bf16*)keys[0], NULL, NULL, (void*)keys[0], 256,
                         NULL) == DS_ESIZE,
          "a short workspace is rejected");
    check(ds_rows_selftest_bounded_wait(NULL, NULL, 1000000ull, NULL) == DS_EINVAL,
          "the self-test needs its buffers");

    if (failures == 0) printf("c consumer: all checks passed\n");
    return failures == 0 ? 0 : 1;
}
