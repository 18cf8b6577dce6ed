/* A plain C99 user of include/gemm.h: compiled and run by the CPU tests to
 * check that the header is C (no C++ types in any signature) and that the
 * library links and answers host-only queries.  With the test-only simulated
 * device it plans the bf16 8192^3 + bias + GELU(tanh) product and prints the
 * plan; it never launches work. */
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include "gemm.h"

int main(void) {
    gemm_plan_t plan;
    gemm_status_t st;
    const uintptr_t base = (uintptr_t)1 << 24; /* stand-in address: planning reads its alignment */
    void* p = (void*)base;

    if (strcmp(gemm_status_string(GEMM_ERR_WORKSPACE), "GEMM_ERR_WORKSPACE") != 0) return 2;
    if (gemm_set_option(GEMM_OPT_TEST_SIM_SMS, 152) != GEMM_OK) return 3;
    memset(&plan, 0, sizeof plan);
    st = gemm_plan_query(GEMM_DT_BF16, 1, 8192, 8192, 8192, p, 8192, GEMM_ROW_MAJOR, 0,
                         p, 8192, GEMM_COL_MAJOR, 0, p, 8192, GEMM_ROW_MAJOR, 0, GEMM_DT_BF16,
                         1.0f, 0.0f, (const float*)p, GEMM_EPI_BIAS_GELU_TANH, 0, 0, &plan);
    if (st != GEMM_OK) return 4;
    printf("kernel=%d block_m=%d block_n=%d block_k=%d stages=%d grid=%d cta_pair=%d "
           "workspace=%lld\n", (int)plan.kernel, (int)plan.block_m, (int)plan.block_n,
           (int)plan.block_k, (int)plan.stages, (int)plan.grid, (int)plan.cta_pair,
           (long long)plan.workspace_bytes);
    printf("workspace_size=%llu\n",
           (unsigned long long)gemm_workspace_size(GEMM_DT_BF16, 1, 256, 256, 65536, 0));
    gemm_set_option(GEMM_OPT_TEST_SIM_SMS, 0);
    return 0;
}
