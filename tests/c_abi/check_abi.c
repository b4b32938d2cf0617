/* A plain C caller of the library's C ABI (include/moe.h). Runs without a GPU: every call
 * below is a size query, a status string, or a call that host validation refuses before
 * anything is launched (the fake addresses are never dereferenced). Exit status 0 when every
 * check holds; otherwise the first failing check is printed. */
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include "moe.h"

#define CHECK(cond)                                                     \
    do {                                                                \
        if (!(cond)) {                                                  \
            fprintf(stderr, "check failed (line %d): %s\n", __LINE__, #cond); \
            return 1;                                                   \
        }                                                               \
    } while (0)

int main(void) {
    const moe_dims full = {64, 2048, 256, 8, 512, 512, 0};
    const moe_dims bad_k = {64, 2048, 256, 9, 512, 512, 0};
    const moe_dims bad_flags = {64, 2048, 256, 8, 512, 512, 2};
    const moe_dims none = {0, 2048, 256, 8, 512, 512, 0};
    char* A = (char*)(uintptr_t)0x10000000u; /* 16-byte aligned, never dereferenced */
    moe_weights w;
    w.router_w = A + 0x1000;
    w.router_b = NULL;
    w.gate_up = A + 0x2000;
    w.down = A + 0x3000;
    w.shared_gate_up = A + 0x4000;
    w.shared_down = A + 0x5000;
    w.shared_gate = A + 0x6000;

    const size_t ws = moe_workspace_size(&full);
    CHECK(ws > 0);
    CHECK(moe_workspace_size(&bad_k) == 0);
    CHECK(moe_workspace_size(&bad_flags) == ws); /* sizes ignore flags */
    CHECK(moe_expert_shadow_size(&full) == (size_t)256 * (2 * 512 * 2048 + 2048 * 512) * 2);

    CHECK(moe_forward(NULL, A, &w, NULL, A + 0x100000, A + 0x200000, ws, NULL) == MOE_ERR_INVALID_ARG);
    CHECK(moe_forward(&bad_k, A, &w, NULL, A + 0x100000, A + 0x200000, ws, NULL) == MOE_ERR_UNSUPPORTED_SHAPE);
    CHECK(moe_forward(&bad_flags, A, &w, NULL, A + 0x100000, A + 0x200000, ws, NULL) == MOE_ERR_INVALID_ARG);
    CHECK(moe_forward(&full, A + 8, &w, NULL, A + 0x100000, A + 0x200000, ws, NULL) == MOE_ERR_MISALIGNED);
    CHECK(moe_forward(&full, A, &w, NULL, A + 0x100000, A + 0x200000, ws - 256, NULL) == MOE_ERR_WORKSPACE_TOO_SMALL);
    CHECK(moe_forward(&none, NULL, &w, NULL, NULL, NULL, 0, NULL) == MOE_OK); /* T = 0: nothing to do */
    CHECK(moe_route(&full, A, &w, NULL, A, A, A, A, A, ws, NULL) == MOE_ERR_INVALID_ARG);
    CHECK(moe_forward_host_experts(&full, A, &w, NULL, A + 0x100000, NULL, 0, A + 0x200000, ws, NULL) ==
          MOE_ERR_INVALID_ARG);
    CHECK(moe_forward_host_io(&full, NULL, &w, NULL, A, A + 0x100000, A + 0x200000, A + 0x400000, ws, NULL) ==
          MOE_ERR_INVALID_ARG); /* no host x */

    CHECK(strncmp(moe_status_string(MOE_OK), "MOE_OK", 6) == 0);
    CHECK(strncmp(moe_status_string(MOE_ERR_MISALIGNED), "MOE_ERR_MISALIGNED", 18) == 0);
    printf("C ABI checks passed (workspace %zu bytes at T=64)\n", ws);
    return 0;
}
