/* Plain C99 use of the library's C ABI: the header compiles as C, and the
 * host-only entry points (partition layout, accounting, status strings) run
 * without a GPU.  Prints one line per result for the test to compare. */
#include <stdint.h>
#include <stdio.h>

#include "zero.h"

int main(void)
{
    zero_layout_t L;
    if (zero_partition_layout(350000017ull, 16u, 15u, 8u, &L) != ZERO_OK)
        return 1;
    printf("layout %llu %llu %llu %llu %llu\n", (unsigned long long)L.shard_elems,
           (unsigned long long)L.begin, (unsigned long long)L.length,
           (unsigned long long)L.padded_elems, (unsigned long long)L.row_pitch);
    for (uint32_t stage = 0; stage <= 3; ++stage)
        printf("bytes %u %llu\n", stage,
               (unsigned long long)zero_model_state_bytes(7500000000ull, 64u, stage, 12u));
    printf("invalid %d\n", (int)zero_partition_layout(10ull, 0u, 0u, 8u, &L));
    printf("status %s\n", zero_status_string(ZERO_ERR_TIMEOUT));
    printf("window %llu\n", (unsigned long long)ZERO_FUSED_WINDOW_ELEMS);
    return 0;
}
