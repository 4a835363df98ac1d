/*
 * The library's host entry points called from plain C99 through include/pa.h
 * alone: the header compiles as C and libpa links and runs without Python.
 * Values from auto-20261007-1900-en (lihaoran.work), "A block table maps
 * logical order to physical storage" (table [5,1,7], b = 4: position 9 is
 * block 7, offset 1) and "How many tail slots remain unused?" (10 tokens in
 * 4-slot blocks: 3 blocks, 2 idle slots).  Prints "ok" and exits 0 on success.
 */
#include <stdio.h>
#include <string.h>

#include "pa.h"

#define CHECK(c)                                                  \
    do {                                                          \
        if (!(c)) {                                               \
            fprintf(stderr, "%s:%d: %s\n", __FILE__, __LINE__, #c); \
            return 1;                                             \
        }                                                         \
    } while (0)

int main(void)
{
    int64_t blocks = 0, unused = 0;
    CHECK(pa_version() > 0);
    CHECK(strlen(pa_status_string(PA_OK)) > 0);
    CHECK(pa_block_layout(10, 4, &blocks, &unused) == PA_OK && blocks == 3 && unused == 2);
    CHECK(pa_block_layout(-1, 4, &blocks, &unused) == PA_ERR_INVALID_ARG);

    const int32_t table[3] = {5, 1, 7};
    const int32_t seq_idx[1] = {0};
    const int64_t pos[1] = {9};
    int64_t slot = -1;
    CHECK(pa_slot_mapping(&slot, table, 1, 3, seq_idx, pos, 1, 4, 8) == PA_OK && slot == 7 * 4 + 1);

    /* a block manager: one sequence of 10 tokens, a fork, copy-on-write on append */
    pa_bm *bm = NULL;
    int32_t a = -1, b = -1, pair[2] = {-1, -1}, n_cow = 0, nb = 0, tab[8];
    int64_t slots[10], ntok = 0;
    CHECK(pa_bm_create(&bm, 8, 4) == PA_OK && bm != NULL);
    CHECK(pa_bm_add_seq(bm, &a) == PA_OK);
    CHECK(pa_bm_append_tokens(bm, a, 10, slots, pair, &n_cow) == PA_OK && n_cow == 0);
    CHECK(pa_bm_get_table(bm, a, tab, 8, &nb, &ntok) == PA_OK && nb == 3 && ntok == 10);
    CHECK(slots[9] == (int64_t)tab[2] * 4 + 1);
    CHECK(pa_bm_fork(bm, a, &b) == PA_OK);
    CHECK(pa_bm_append_tokens(bm, b, 1, slots, pair, &n_cow) == PA_OK && n_cow == 1 && pair[0] == tab[2]);
    pa_bm_destroy(bm);

    /* cascade planning: two sequences sharing two whole blocks */
    const int32_t tables2[2][4] = {{3, 4, 5, -1}, {3, 4, 6, 7}};
    const int32_t lens[2] = {40, 60};
    int32_t ptab[1][4], plen[1], order[1], stab[2][4], slen[2];
    CHECK(pa_cascade_plan(&tables2[0][0], 4, lens, 2, 2, 16, &ptab[0][0], plen, order, &stab[0][0], slen) == PA_OK);
    CHECK(plen[0] == 32 && order[0] == 0 && ptab[0][0] == 3 && ptab[0][1] == 4 && ptab[0][2] == -1);
    CHECK(slen[0] == 8 && slen[1] == 28 && stab[0][0] == 5 && stab[1][0] == 6 && stab[1][1] == 7);

    puts("ok");
    return 0;
}
