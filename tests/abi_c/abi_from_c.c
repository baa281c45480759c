/* Compiled and run by tests/test_abi.py on a machine without a GPU: the header is valid C, the
 * library links from C, and calls with invalid arguments return their status codes before any
 * device work.  No call here reaches a kernel launch. */
#include <stdio.h>
#include <string.h>

#include "swa_b300.h"

static int fails = 0;
#define EXPECT(cond)                                                \
    do {                                                            \
        if (!(cond)) {                                              \
            fprintf(stderr, "line %d: %s\n", __LINE__, #cond);      \
            ++fails;                                                \
        }                                                           \
    } while (0)

int main(void) {
    void* P = (void*)0x10000; /* 16-byte aligned, never dereferenced */
    EXPECT(strcmp(swa_status_string(SWA_OK), "unknown status") != 0);
    EXPECT(strcmp(swa_status_string(99), "unknown status") == 0);
    EXPECT(swa_attn_fwd(NULL, P, P, P, 1, 2, 2, 128, 64, 16, 0.125f, NULL) == SWA_ERR_NULL);
    EXPECT(swa_attn_fwd(P, P, P, P, 1, 3, 2, 128, 64, 16, 0.125f, NULL) == SWA_ERR_SHAPE);
    EXPECT(swa_attn_fwd(P, P, P, P, 1, 2, 2, 128, 96, 16, 0.125f, NULL) == SWA_ERR_UNSUPPORTED);
    EXPECT(strided_attn_fwd(P, P, P, P, 1, 2, 2, 128, 64, 16, 0, 0.125f, NULL) == SWA_ERR_SHAPE);
    EXPECT(diff_attn_fwd(P, P, P, P, P, 0.8f, NULL, 1, 2, 2, 128, 64, 0.125f, NULL) ==
           SWA_ERR_NULL);
    EXPECT(diff_swa_attn_fwd(P, P, P, P, P, 0.8f, NULL, P, 1, 2, 2, 128, 64, 0, 0.125f, NULL) ==
           SWA_ERR_SHAPE);
    EXPECT(global_attn_fwd(P, P, P, P, 1, 2, 2, 128, 64, 16, -1, 0.125f, NULL) == SWA_ERR_SHAPE);
    EXPECT(swa_decode_workspace_bytes(2, 8, 300, 128) > 0);
    EXPECT(swa_decode_workspace_bytes(2, 8, 300, 96) == 0);
    size_t nb = swa_attn_bwd_workspace_bytes(2, 4, 300);
    EXPECT(nb >= 2 * 4 * 300 * 4);
    EXPECT(swa_attn_bwd(P, P, P, P, (const float*)P, P, P, P, P, 2, 4, 2, 300, 64, 50, 0.125f, P,
                        nb - 1, NULL) == SWA_ERR_TOO_LARGE);
    EXPECT(swa_attn_bwd(P, P, P, P, NULL, P, P, P, P, 2, 4, 2, 300, 64, 50, 0.125f, P, nb, NULL) ==
           SWA_ERR_NULL);
    if (fails == 0) printf("abi from C: ok\n");
    return fails == 0 ? 0 : 1;
}
