/* include/pkv.h used from plain C99 (built with -std=c99 -pedantic -Werror by
 * tests/test_native_host.py): the header compiles as C, and the block
 * manager's calls work from C with no C++ on the caller's side.  Host calls
 * only; the device entry points are only referenced. */
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "pkv.h"

#define EXPECT(c)                                                   \
    do {                                                            \
        if (!(c)) {                                                 \
            printf("FAIL %s:%d: %s\n", __FILE__, __LINE__, #c);     \
            return 1;                                               \
        }                                                           \
    } while (0)

int main(void) {
    /* a pool of 8 blocks of 4 slots; two sequences, one forked */
    pkv_alloc_t *a = NULL, *b = NULL;
    int32_t seqs[3], tables[3 * 4], lens[3], pairs[2 * 3];
    int64_t slots[3];
    int n_cow = -1, child = -1, i;
    size_t bytes = 0;
    void *blob;
    /* every device entry point is declared with C linkage */
    int (*decode)(void *, const void *, const void *, const void *, const int32_t *, int, const int32_t *, int,
                  int, int, int, int, int, float, int, void *, size_t, int32_t *, pkv_stream_t) =
        pkv_paged_attention_decode;
    EXPECT(decode != NULL);

    EXPECT(pkv_alloc_create(8, 4, NULL, &a) == PKV_OK);
    EXPECT(pkv_seq_new(a, &seqs[0]) == PKV_OK && seqs[0] == 0);
    EXPECT(pkv_seq_new(a, &seqs[1]) == PKV_OK && seqs[1] == 1);
    EXPECT(pkv_append_tokens(a, seqs[0], 6, NULL, NULL, &n_cow) == PKV_OK && n_cow == 0);
    EXPECT(pkv_fork(a, seqs[0], &child) == PKV_OK && child == 2);
    seqs[2] = child;
    /* one token each, in batch order: seq 0 copies the shared partial block 1
     * to block 2, seq 1 takes block 3, and the fork, now block 1's only
     * holder, writes in place */
    EXPECT(pkv_append_batch(a, seqs, 3, slots, pairs, &n_cow) == PKV_OK);
    EXPECT(n_cow == 1 && pairs[0] == 1 && pairs[1] == 2);
    EXPECT(slots[0] == 2 * 4 + 2 && slots[1] == 3 * 4 + 0 && slots[2] == 1 * 4 + 2);
    EXPECT(pkv_export_tables(a, seqs, 3, tables, 4, lens) == PKV_OK);
    EXPECT(lens[0] == 7 && lens[1] == 1 && lens[2] == 7);
    EXPECT(tables[0] == 0 && tables[1] == 2 && tables[2] == -1 && tables[4] == 3);
    EXPECT(tables[8] == 0 && tables[9] == 1);

    /* checkpoint round trip */
    EXPECT(pkv_alloc_save(a, NULL, 0, &bytes) == PKV_OK && bytes > 0);
    blob = malloc(bytes);
    EXPECT(blob != NULL);
    EXPECT(pkv_alloc_save(a, blob, bytes, &bytes) == PKV_OK);
    EXPECT(pkv_alloc_load(blob, bytes, &b) == PKV_OK);
    memset(tables, 0, sizeof tables);
    EXPECT(pkv_export_tables(b, seqs, 3, tables, 4, lens) == PKV_OK);
    EXPECT(lens[0] == 7 && tables[1] == 2 && tables[9] == 1);
    EXPECT(pkv_alloc_load(blob, bytes - 1, &b) == PKV_ERR_INVALID_ARG);
    free(blob);

    /* errors come back as codes, with names */
    EXPECT(pkv_fork(a, 99, &child) == PKV_ERR_NOT_FOUND);
    EXPECT(strcmp(pkv_status_string(PKV_ERR_NOT_FOUND), "PKV_ERR_NOT_FOUND") == 0);
    for (i = 0; i < 3; ++i) EXPECT(pkv_release(a, seqs[i], NULL) == PKV_OK);
    {
        int nfree = 0;
        EXPECT(pkv_num_free(a, &nfree) == PKV_OK && nfree == 8);
    }
    pkv_alloc_destroy(a);
    pkv_alloc_destroy(b);
    printf("c99 header ok\n");
    return 0;
}
