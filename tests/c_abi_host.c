/*
 * A plain C99 caller of the library's host-side entry points, built and run
 * by tests/test_abi.py (no GPU): it includes include/pkv.h as C, links
 * libpkv.so and checks the slot-mapping and prefix-group helpers, the block
 * allocator's lifecycle and the argument checks that fail before any launch.
 * Exit status 0 = every check held; otherwise the failing line is printed.
 */
#include <stdio.h>
#include <string.h>

#include "pkv.h"

static int failures = 0;
#define CHECK(cond)                                                         \
    do {                                                                    \
        if (!(cond)) {                                                      \
            fprintf(stderr, "c_abi_host.c:%d: check failed: %s\n", __LINE__, #cond); \
            ++failures;                                                     \
        }                                                                   \
    } while (0)

static void slot_mapping(void)
{
    /* two rows of a 8-block pool, block size 16; row 1 has no second block */
    const int32_t tables[2][2] = {{3, 7}, {5, -1}};
    const int32_t rows[4] = {0, 1, 0, 1};
    const int32_t pos[4] = {20, 3, 0, 17};
    int32_t slots[4] = {0, 0, 0, 0};
    /* the missing entry (row 1, position 17) gets -1 and fails the call */
    CHECK(pkv_slot_mapping_host(&tables[0][0], 2, 2, 8, rows, pos, 4, 16, slots) ==
          PKV_ERR_INVALID_ARG);
    CHECK(slots[0] == 7 * 16 + 4 && slots[1] == 5 * 16 + 3 && slots[2] == 3 * 16 && slots[3] == -1);
    CHECK(pkv_slot_mapping_host(&tables[0][0], 2, 2, 8, rows, pos, 3, 16, slots) == PKV_OK);
    {
        /* the debug check: slots 116, 83, 48 are distinct and inside the pool */
        int32_t bad = 7;
        const int32_t twice[3] = {48, -1, 48};
        CHECK(pkv_slot_mapping_check_host(slots, 3, 8, 16, &bad) == PKV_OK && bad == -1);
        CHECK(pkv_slot_mapping_check_host(twice, 3, 8, 16, &bad) == PKV_ERR_INVALID_ARG &&
              bad == 2);
    }
}

static void prefix_groups(void)
{
    /* rows 0 and 1 share blocks 2, 4; row 2 starts elsewhere */
    const int32_t tables[3][3] = {{2, 4, 6}, {2, 4, 1}, {3, 0, 5}};
    const int32_t lens[3] = {40, 45, 30};
    int32_t group_of_row[3] = {9, 9, 9};
    int32_t prefix_blocks[3] = {9, 9, 9};
    CHECK(pkv_prefix_groups_host(&tables[0][0], 3, lens, 3, 16, group_of_row, prefix_blocks) == 1);
    CHECK(group_of_row[0] == 0 && group_of_row[1] == 0 && group_of_row[2] == -1);
    CHECK(prefix_blocks[0] == 2);
    /* a row whose second block is not full yet keeps the prefix to one block */
    {
        const int32_t short_lens[3] = {40, 20, 30};
        CHECK(pkv_prefix_groups_host(&tables[0][0], 3, short_lens, 3, 16, group_of_row,
                                     prefix_blocks) == 1);
        CHECK(prefix_blocks[0] == 1);
    }
}

static void allocator(void)
{
    int32_t tokens[40];
    int32_t table[4];
    int32_t n = 0, cached = -1, nb = 0, nfree = 0, ncached = 0, grows = 0;
    int i;
    pkv_allocator *a;
    int32_t ra, rb;
    for (i = 0; i < 40; ++i) tokens[i] = 1000 + i;
    a = pkv_allocator_create(16, 4, 16);
    CHECK(a != NULL);
    if (a == NULL) return;

    /* request a: nothing cached; 41 tokens take blocks 0, 1, 2 (lowest first) */
    ra = pkv_allocator_begin(a);
    CHECK(pkv_allocator_find_cached_prefix(a, ra, tokens, 40, NULL, &cached) == PKV_OK);
    CHECK(cached == 0);
    CHECK(pkv_allocator_reserve(a, ra, 41) == PKV_OK);
    CHECK(pkv_allocator_publish(a, ra, tokens, 40, NULL) == PKV_OK);  /* 2 full blocks */
    CHECK(pkv_allocator_table(a, ra, table, 4, &n) == PKV_OK);
    CHECK(n == 3 && table[0] == 0 && table[1] == 1 && table[2] == 2);

    /* request b, same prompt: its two full blocks are shared, one new block */
    rb = pkv_allocator_begin(a);
    CHECK(pkv_allocator_find_cached_prefix(a, rb, tokens, 40, NULL, &cached) == PKV_OK);
    CHECK(cached == 32);
    CHECK(pkv_allocator_reserve(a, rb, 41) == PKV_OK);
    CHECK(pkv_allocator_table(a, rb, table, 4, &n) == PKV_OK);
    CHECK(n == 3 && table[0] == 0 && table[1] == 1 && table[2] == 3);
    CHECK(pkv_allocator_refcount(a, 0) == 2 && pkv_allocator_refcount(a, 3) == 1);

    /* releases: shared blocks drop a reference; published ones end cache-only */
    CHECK(pkv_allocator_release(a, ra) == PKV_OK);
    CHECK(pkv_allocator_refcount(a, 0) == 1 && pkv_allocator_refcount(a, 2) == 0);
    CHECK(pkv_allocator_stats(a, &nb, &nfree, &ncached, &grows) == PKV_OK);
    CHECK(nb == 4 && nfree == 1 && ncached == 0 && grows == 0);
    CHECK(pkv_allocator_release(a, rb) == PKV_OK);
    CHECK(pkv_allocator_stats(a, &nb, &nfree, &ncached, &grows) == PKV_OK);
    CHECK(nb == 4 && nfree == 2 && ncached == 2);

    /* 5 blocks more than the 4 held: the pool grows (doubles) before evicting */
    ra = pkv_allocator_begin(a);
    CHECK(pkv_allocator_reserve(a, ra, 5 * 16) == PKV_OK);
    CHECK(pkv_allocator_stats(a, &nb, &nfree, &ncached, &grows) == PKV_OK);
    CHECK(nb == 8 && grows == 1);
    CHECK(pkv_allocator_release(a, 12345) == PKV_ERR_INVALID_ARG);  /* no such request */
    pkv_allocator_destroy(a);
}

static void argument_checks(void)
{
    pkv_pool pool;
    memset(&pool, 0, sizeof(pool));
    CHECK(paged_kv_append(NULL, NULL, 1, NULL, NULL, NULL, NULL) == PKV_ERR_INVALID_ARG);
    pool.num_blocks = 16;
    pool.block_size = 16;
    pool.num_kv_heads = 2;
    pool.head_dim = 64;
    pool.dtype = PKV_BF16;
    /* pools with no memory behind them are refused before any launch */
    CHECK(paged_kv_append(&pool, NULL, 1, NULL, NULL, NULL, NULL) == PKV_ERR_INVALID_ARG);
    CHECK(pkv_status_string(PKV_OK) != NULL && pkv_status_string(PKV_ERR_UNSUPPORTED) != NULL);
    CHECK(pkv_version() != NULL && strlen(pkv_version()) > 0);
}

int main(void)
{
    slot_mapping();
    prefix_groups();
    allocator();
    argument_checks();
    if (failures == 0) printf("c_abi_host: ok\n");
    return failures == 0 ? 0 : 1;
}
