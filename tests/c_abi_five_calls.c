/* Compiled against include/chunk_attention.h and linked with
 * libchunk_attention.so by tests/test_capi_signatures.py: the five calls of
 * the problem statement (create a pool, insert with prefix matching, build
 * the per-step schedule, attend, remove) with exactly the declared
 * signatures, so the C compiler checks every argument type.
 *
 * Host-only pool (kv_dev NULL): nothing touches a GPU, so the decode call
 * must answer CA_ERR_INVALID; the trie and schedule still work.  Two
 * sequences share a 2-chunk prefix [ChunkAttention §3.1: sequences with a
 * common prompt share its chunks], so the second insert matches 32 tokens
 * and the schedule has two chunk-first rows [§3.2].
 *
 * Exit status 0 when every expectation holds; otherwise the number of the
 * failed check. */
#include <stdio.h>

#include "chunk_attention.h"

#define EXPECT(n, cond)                                          \
    do {                                                         \
        if (!(cond)) {                                           \
            fprintf(stderr, "check %d failed: %s\n", n, #cond);  \
            return n;                                            \
        }                                                        \
    } while (0)

int main(void) {
    ca_pool_config cfg = {1, 2, 64, 16, 32, 0u};   /* L, H, D, c, slots, flags */
    ca_pool* pool = NULL;
    EXPECT(1, ca_pool_create(&cfg, NULL, 0, &pool) == CA_OK && pool != NULL);

    int32_t a[40], b[40];
    for (int i = 0; i < 40; ++i) {
        a[i] = i;                     /* 32 shared tokens, then a's own     */
        b[i] = i < 32 ? i : 1000 + i; /* the same 32, then b's own          */
    }
    int32_t shared = -1;
    EXPECT(2, ca_insert_tokens(pool, 7, a, 40, NULL, NULL, NULL, &shared) == CA_OK && shared == 0);
    EXPECT(3, ca_insert_tokens(pool, 9, b, 40, NULL, NULL, NULL, &shared) == CA_OK && shared == 32);
    EXPECT(4, ca_insert_tokens(pool, 9, b, 40, NULL, NULL, NULL, &shared) == CA_ERR_EXISTS);

    const int64_t batch[2] = {9, 7};
    ca_sched* sched = NULL;
    EXPECT(5, ca_build_schedule(pool, batch, 2, &sched, NULL) == CA_OK && sched != NULL);
    int32_t counts[6];
    EXPECT(6, ca_sched_counts(sched, counts) == CA_OK);
    EXPECT(7, counts[0] == 2 && counts[1] == 2 && counts[2] == 1 && counts[3] == 2);
    size_t ws = 0;
    EXPECT(8, ca_workspace_bytes(sched, &ws) == CA_OK && ws > 0);

    /* A host-only pool has no device memory to attend over. */
    EXPECT(9, ca_decode_attention(pool, sched, 0, NULL, NULL, 0.125f, NULL, 0, NULL) == CA_ERR_INVALID);

    EXPECT(10, ca_remove_seq(pool, 7) == CA_OK);
    EXPECT(11, ca_remove_seq(pool, 7) == CA_ERR_NOT_FOUND);
    /* The tree changed: the schedule is stale until rebuilt. */
    const int64_t one[1] = {9};
    EXPECT(12, ca_build_schedule(pool, one, 1, &sched, NULL) == CA_OK);
    EXPECT(13, ca_sched_counts(sched, counts) == CA_OK && counts[1] == 0 && counts[3] == 3);
    ca_stats st;
    EXPECT(14, ca_pool_stats(pool, &st) == CA_OK && st.live_slots == 3 && st.live_seqs == 1);
    EXPECT(15, ca_remove_seq(pool, 9) == CA_OK);
    EXPECT(16, ca_pool_stats(pool, &st) == CA_OK && st.live_slots == 0 && st.free_slots == 32);
    EXPECT(17, ca_sched_destroy(sched) == CA_OK && ca_pool_destroy(pool) == CA_OK);
    printf("five calls ok\n");
    return 0;
}
