/* A C99 client of include/pa.h: the header compiles as strict C and the
 * library links and answers from C.  Only host-side entry points are called
 * (the block manager, version and status strings, and a decode call that the
 * host rejects before any CUDA call), so no GPU is needed.  Prints "ok" and
 * exits 0 when every check holds; otherwise prints each failure. */
#include "pa.h"

#include <stdio.h>
#include <string.h>

static int failures = 0;

#define CHECK(cond)                                                  \
    do {                                                             \
        if (!(cond)) {                                               \
            printf("failed: %s (line %d)\n", #cond, __LINE__);       \
            ++failures;                                              \
        }                                                            \
    } while (0)

int main(void) {
    const int codes[] = {PA_OK, PA_FAIL_NO_BLOCKS, PA_ERR_INVALID_ARG, PA_ERR_UNSUPPORTED, PA_ERR_MISALIGNED,
                         PA_ERR_CUDA, PA_ERR_WORKSPACE, PA_ERR_UNKNOWN_SEQ, PA_ERR_DUPLICATE_SEQ, PA_ERR_SWAPPED};
    size_t i;
    const char* v = pa_version();
    CHECK(v != NULL && strlen(v) > 0);
    for (i = 0; i < sizeof(codes) / sizeof(codes[0]); ++i) {
        const char* s = pa_status_string(codes[i]);
        CHECK(s != NULL && strlen(s) > 0);
    }

    /* A pool of 8 blocks of 4 positions: a fresh manager hands out 0, 1, 2, ... */
    {
        pa_alloc_t* a = pa_alloc_create(8, 4);
        pa_alloc_stats_t st;
        int64_t slot = -1;
        int32_t src = -1, dst = -1, table[8], pairs[16];
        int n = 0;
        const int64_t out_seqs[1] = {2};
        CHECK(a != NULL);
        CHECK(pa_alloc_create(0, 4) == NULL);
        CHECK(pa_alloc_sequence(a, 1, 6) == PA_OK);                /* blocks 0, 1 */
        CHECK(pa_alloc_sequence(a, 1, 3) == PA_ERR_DUPLICATE_SEQ);
        CHECK(pa_alloc_fork(a, 1, 2) == PA_OK);                    /* both blocks shared */
        CHECK(pa_alloc_ref_count(a, 0) == 2 && pa_alloc_ref_count(a, 1) == 2);
        /* position 6 lands in the shared, partly filled tail: it is cloned first */
        CHECK(pa_alloc_append_slot(a, 1, &slot, &src, &dst) == PA_OK);
        CHECK(src == 1 && dst == 2 && slot == 2 * 4 + 2);
        CHECK(pa_alloc_block_table(a, 1, table, 8, &n) == PA_OK && n == 2 && table[0] == 0 && table[1] == 2);
        CHECK(pa_alloc_block_table(a, 2, table, 8, &n) == PA_OK && n == 2 && table[0] == 0 && table[1] == 1);
        CHECK(pa_alloc_get_stats(a, &st) == PA_OK);
        CHECK(st.num_blocks == 8 && st.num_used == 3 && st.num_free == 5 && st.num_seqs == 2);
        CHECK(st.num_cow_copies == 1 && st.num_context_tokens == 7 + 6 && st.num_swap_outs == 0);
        CHECK(pa_alloc_get_stats(a, NULL) == PA_ERR_INVALID_ARG);
        /* swap sequence 2 out: its two device blocks go to host blocks */
        CHECK(pa_alloc_enable_swap(a, 4) == PA_OK);
        CHECK(pa_alloc_swap_out(a, out_seqs, 1, pairs, 8, &n) == PA_OK && n == 2);
        CHECK(pa_alloc_is_swapped(a, 2) == 1 && pa_alloc_is_swapped(a, 1) == 0);
        CHECK(pa_alloc_get_stats(a, &st) == PA_OK && st.num_swapped == 1 && st.num_swap_outs == 1);
        CHECK(pa_alloc_append_slot(a, 2, &slot, &src, &dst) == PA_ERR_SWAPPED);
        CHECK(pa_alloc_free(a, 2) == PA_OK && pa_alloc_free(a, 1) == PA_OK);
        CHECK(pa_alloc_num_free(a) == 8);
        pa_alloc_destroy(a);
        pa_alloc_destroy(NULL);
    }

    /* a device entry point rejects a bad argument on the host, before any CUDA call */
    CHECK(pa_decode(NULL, PA_DTYPE_BF16, NULL, NULL, NULL, NULL, NULL, 16, 0.1f, 32, 8, 128, -1, 8, 64, 128, 0, NULL,
                    0, NULL, NULL) == PA_ERR_INVALID_ARG);

    if (failures == 0) printf("ok\n");
    return failures == 0 ? 0 : 1;
}
