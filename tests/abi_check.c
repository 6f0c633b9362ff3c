/* A C99 caller of the g3s C ABI.  It includes include/g3s.h alone (no CUDA
 * or C++ header), links against libg3s.so and calls the entry points that
 * need no GPU, printing what tests/test_c_abi.py compares with the Python
 * binding.  Test infrastructure only. */
#include <stdio.h>

#include "g3s.h"

int main(void) {
    g3s_plan_options o;
    g3s_plan_options_init(&o);
    size_t bytes = 0;
    g3s_status st = g3s_plan_workspace_size(2000000, 100717572, 4, 32, G3S_BF16, G3S_STANDARD, &o, &bytes);
    printf("version %s\n", g3s_version());
    printf("headline %s %zu\n", g3s_status_string(st), bytes);
    st = g3s_plan_workspace_size(40851, 560593, 8, 64, G3S_BF16, G3S_STANDARD, NULL, &bytes);
    printf("batched %s %zu\n", g3s_status_string(st), bytes);
    st = g3s_plan_workspace_size(100, 1000, 4, 48, G3S_BF16, G3S_STANDARD, NULL, &bytes);
    printf("bad_head_dim %s\n", g3s_status_string(st));
    const int unsupported = st == G3S_ERR_UNSUPPORTED;
    printf("struct_sizes %zu %zu\n", sizeof(g3s_plan_options), sizeof(g3s_plan_stats));
    printf("defaults %d %d %d %d %d\n", (int)o.tile_density_milli, (int)o.tile_pool_density_milli,
           (int)o.tile_split_density_milli, (int)o.tile_split_parallel, (int)o.small_graph_rows);
    printf("error_detail %s\n", g3s_last_error());
    return unsupported ? 0 : 1;
}
