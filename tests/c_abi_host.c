/* A plain C program against include/zero.h and libzero_shard.so, using the entry points
 * that need no GPU: the partition/ledger, the workspace size, the per-tensor segment map
 * and the status texts; and the step state's layout as the header defines it (one line
 * per field, which the test compares with the Python binding's).  Built and run by
 * tests/test_c_abi.py; prints one line per check and exits non-zero on the first
 * failure. */
#include <stddef.h>
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include "zero.h"

static int fail(const char* what)
{
    printf("FAIL %s\n", what);
    return 1;
}

int main(void)
{
    /* the 8-parameter, 4-GPU example of the ZeRO walkthrough: two parameters per rank */
    zero_layout_t L;
    if (zero_partition(8, 4, 2, 1, 0, &L) != ZERO_OK)
        return fail("zero_partition");
    if (L.shard != 2 || L.psi_padded != 8 || L.pad != 0 || L.n_ranks != 4)
        return fail("layout");
    /* stage 2 ledger: 2 bytes of weights for all, 2 + 12 bytes per own parameter */
    if (L.bytes_per_rank[2] != 2 * 8 + 14 * 2)
        return fail("ledger");
    if (zero_workspace_bytes(&L) != (size_t)L.n_tiles * 8)
        return fail("workspace");
    printf("partition psi=8 N=4: S=%llu, stage-2 bytes per rank %llu\n",
           (unsigned long long)L.shard, (unsigned long long)L.bytes_per_rank[2]);

    /* tensors of 3 and 5 parameters: pieces (tensor, rank, offset in tensor, count) */
    const uint64_t sizes[2] = {3, 5};
    uint64_t n = 0;
    if (zero_segment_map(&L, sizes, 2, NULL, 0, &n) != ZERO_OK || n != 5)
        return fail("segment count");
    zero_segment_t seg[5];
    if (zero_segment_map(&L, sizes, 2, seg, 5, &n) != ZERO_OK)
        return fail("segment map");
    const uint64_t want[5][5] = {{0, 0, 0, 0, 2}, {0, 1, 2, 0, 1}, {1, 1, 0, 1, 1},
                                 {1, 2, 1, 0, 2}, {1, 3, 3, 0, 2}};
    for (int i = 0; i < 5; ++i) {
        const uint64_t got[5] = {seg[i].tensor, seg[i].rank, seg[i].tensor_offset,
                                 seg[i].shard_offset, seg[i].count};
        if (memcmp(got, want[i], sizeof got) != 0)
            return fail("segment piece");
    }
    printf("segment map: 5 pieces as expected\n");

    if (zero_partition(0, 4, 2, 1, 0, &L) != ZERO_EINVAL)
        return fail("empty model rejected");
    if (strlen(zero_strerror(ZERO_EINVAL)) == 0)
        return fail("strerror");
#define FIELD(f) printf("state %s %zu\n", #f, offsetof(zero_step_state_t, f))
    FIELD(sumsq); FIELD(norm); FIELD(clip_coef); FIELD(loss_scale); FIELD(inv_scale);
    FIELD(step_size); FIELD(rbc2); FIELD(decay); FIELD(overflow); FIELD(skip); FIELD(t);
    FIELD(good_steps); FIELD(growth_interval); FIELD(dynamic); FIELD(n_ranks); FIELD(n_steps);
    FIELD(n_skipped); FIELD(error); FIELD(arrivals); FIELD(inv_scale_used);
    FIELD(launch_arrivals); FIELD(applied_c); FIELD(adamw_next_chunk); FIELD(adamw_done);
    FIELD(reserved);
#undef FIELD
    printf("state_size %zu\n", sizeof(zero_step_state_t));
    printf("ok\n");
    return 0;
}
