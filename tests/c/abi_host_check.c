/* A plain C99 caller of libgcl: includes the public header, links the library and
 * exercises the host-side parts of the ABI (sizes, status strings, argument checks).
 * Nothing here touches a GPU, so it runs on any machine that has the CUDA runtime. */
#include <stdio.h>
#include <string.h>

#include "gcl.h"

static int fails = 0;
#define CHECK(cond)                                                   \
    do {                                                              \
        if (!(cond)) {                                                \
            fprintf(stderr, "check failed: %s (line %d)\n", #cond, __LINE__); \
            ++fails;                                                  \
        }                                                             \
    } while (0)

int main(void) {
    /* NT_max = ceil(T_max / BT) + N_max - 1 */
    CHECK(gcl_nt_max(65536, 64, 64) == 1087);
    CHECK(gcl_nt_max(4096, 1, 64) == 64);
    CHECK(gcl_nt_max(100, 3, 32) == 6);
    CHECK(strcmp(gcl_status_string(GCL_OK), "GCL_OK") == 0);

    /* NULL argument structs are rejected before anything is enqueued */
    CHECK(gdn_chunk_fwd(NULL, NULL) == GCL_ERR_INVALID_ARG);
    CHECK(kda_chunk_bwd(NULL, NULL) == GCL_ERR_INVALID_ARG);
    CHECK(causal_conv1d_fwd(NULL, NULL) == GCL_ERR_INVALID_ARG);

    /* an unsupported head size is reported with a reason */
    gcl_fwd_args a;
    memset(&a, 0, sizeof a);
    a.q = a.k = a.v = (const void *)(size_t)(1u << 20);
    a.g = (const float *)(size_t)(1u << 20);
    a.beta = (const void *)(size_t)(1u << 20);
    a.cu_seqlens = (const int32_t *)(size_t)(1u << 20);
    a.o = (void *)(size_t)(1u << 20);
    a.t_max = 128;
    a.n_max = 1;
    a.H = 1;
    a.K = 96;
    a.V = 128;
    a.bt = 64;
    a.scale = 1.0f;
    a.dtype = GCL_BF16;
    CHECK(gdn_chunk_fwd(&a, NULL) == GCL_ERR_UNSUPPORTED);
    CHECK(strlen(gcl_last_error()) > 0);

    /* workspace queries are pure functions of the sizes */
    a.K = 128;
    CHECK(gcl_fwd_workspace_min_bytes(&a) > 0);
    CHECK(gcl_fwd_workspace_bytes(&a) >= gcl_fwd_workspace_min_bytes(&a));

    if (fails == 0) printf("c abi ok\n");
    return fails == 0 ? 0 : 1;
}
