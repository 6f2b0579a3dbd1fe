/*
 * Plain C99 use of the library's C ABI (include/kvq.h), host-only calls
 * that need no GPU: pool sizes, status strings, arguments refused before
 * anything is launched, and one residency plan of a streamed pool.
 * Built and run by tests/test_c_abi.py, which checks what it prints.
 */
#include <stdio.h>
#include <string.h>

#include "kvq.h"

int main(void) {
    kvq_cache c;
    int s;
    int32_t slot_of[6], block_of[3], slots[4], src[3], dst[3];
    const int32_t table[4] = {4, 1, 5, 2};
    const int32_t lens[1] = {40};
    int64_t last[3] = {0, 0, 0}, clock = 0;
    int n_fetch = -1, n_hits = -1;

    printf("block_bytes %lu %lu %lu\n", (unsigned long)kvq_block_bytes(KVQ_F16, 8, 128, 256),
           (unsigned long)kvq_block_bytes(KVQ_Q8, 8, 128, 256),
           (unsigned long)kvq_block_bytes(KVQ_K8V4, 2, 256, 256));
    for (s = KVQ_OK; s <= KVQ_ERR_CUDA; ++s)
        if (kvq_status_string(s) == NULL || kvq_status_string(s)[0] == '\0') return 2;

    /* an int8 cache without its arrays: refused, nothing launched */
    memset(&c, 0, sizeof c);
    c.fmt = KVQ_Q8;
    c.n_kv_heads = 1;
    c.head_dim = 64;
    c.block_size = 16;
    c.n_blocks = 1;
    printf("append %d\n", (int)kvq_append(&c, NULL, NULL, 1, NULL, NULL, NULL, 1, 1, NULL));
    printf("decode %d\n", (int)kvq_decode_attn(&c, NULL, 1, 1, 4, NULL, 16, NULL, 1, 0.125f, NULL,
                                                NULL, 0, NULL));
    printf("workspace %lu\n", (unsigned long)kvq_decode_workspace_bytes(NULL, 1, 1, 4, 16));

    /* 6 host blocks, a window of 3 slots; one sequence of 40 cells at block
     * size 16 reads blocks 4, 1, 5 (entry 3 of its row is past its cells) */
    for (s = 0; s < 6; ++s) slot_of[s] = -1;
    for (s = 0; s < 3; ++s) block_of[s] = -1;
    s = (int)kvq_stream_plan(6, 3, slot_of, block_of, last, &clock, table, 1, 4, lens, 16, slots,
                             src, dst, &n_fetch, &n_hits);
    printf("plan %d fetch %d hits %d\n", s, n_fetch, n_hits);
    printf("pairs %d:%d %d:%d %d:%d\n", src[0], dst[0], src[1], dst[1], src[2], dst[2]);
    printf("slots %d %d %d %d\n", slots[0], slots[1], slots[2], slots[3]);
    /* the same call again: every block is resident */
    s = (int)kvq_stream_plan(6, 3, slot_of, block_of, last, &clock, table, 1, 4, lens, 16, slots,
                             src, dst, &n_fetch, &n_hits);
    printf("again %d fetch %d hits %d\n", s, n_fetch, n_hits);
    return 0;
}
