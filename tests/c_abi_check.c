/* A plain C program against include/ts.h and libts.so: the C ABI is usable
 * without Python or torch.  Host-only calls (tree mask, workspace size,
 * argument validation) run without a GPU; the program prints one line per
 * check and exits non-zero on the first failure. */
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include "ts.h"

#define CHECK(cond, what)                                   \
    do {                                                    \
        if (!(cond)) {                                      \
            printf("FAIL %s\n", what);                      \
            return 1;                                       \
        }                                                   \
        printf("ok %s\n", what);                            \
    } while (0)

int main(void) {
    CHECK(strstr(ts_version(), "sm_103a") != NULL, "version names sm_103a");

    /* tree 0 <- {1, 2}, 1 <- 3; row 3 sees 0, 1 and itself */
    const int32_t parent[4] = {-1, 0, 0, 1};
    uint64_t mask[8];
    CHECK(ts_tree_mask_from_parents(parent, 4, mask) == TS_OK, "mask of a small tree");
    CHECK(mask[0] == 0x1 && mask[2] == 0x3 && mask[4] == 0x5 && mask[6] == 0xb, "ancestor-or-self bits");
    CHECK(mask[1] == 0 && mask[7] == 0, "upper words empty");

    const int32_t bad[2] = {-1, 1};
    CHECK(ts_tree_mask_from_parents(bad, 2, mask) == TS_ERR_INVALID_ARG, "self-parent rejected");
    CHECK(strlen(ts_last_error()) > 0, "error message set");

    CHECK(ts_tree_attn_workspace_bytes(120, 40, 8, 128, 102400) > 0, "verify workspace is split");
    CHECK(ts_tree_attn_workspace_bytes(120, 40, 7, 128, 102400) == 0, "Hq % Hkv != 0 needs none");

    /* validation happens before any device work: fake aligned pointers */
    void *P = (void *)(uintptr_t)0x10000;
    ts_status st = ts_tree_attn(P, P, P, 5000, 4096, 40, 4, 1, 96, 0.125f, (const uint64_t *)P, P, NULL, NULL, 0,
                                P, (size_t)1 << 30, NULL);
    CHECK(st == TS_ERR_UNSUPPORTED, "head dim 96 unsupported");
    st = ts_commit_path(P, P, 100, 4096, 120, 8, 128, (int32_t *)P, (const int32_t *)P, NULL);
    CHECK(st == TS_ERR_INVALID_ARG, "commit with ld_kv < N + T rejected");
    return 0;
}
