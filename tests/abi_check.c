/* A plain C99 caller of libmoe: include/moe.h must compile as C (not only as
 * C++), and the host-only entry points must behave as declared when called
 * from C. Needs no GPU. Built and run by test_abi_c.py; argv[1] names a file
 * that does not exist. */
#include <stdio.h>
#include <string.h>

#include "moe.h"

#define CHECK(c)                                                             \
    do {                                                                     \
        if (!(c)) {                                                          \
            fprintf(stderr, "check failed at line %d: %s\n", __LINE__, #c); \
            return 1;                                                        \
        }                                                                    \
    } while (0)

int main(int argc, char** argv) {
    const moe_shapes tiny = {512, 16, 2, 256, 512, 0};
    const int32_t toy[7] = {1, 2, 1, 3, 4, 1, 2};
    const int32_t pair_ids[6] = {3, 1, 3, 0, 1, 3};
    const int32_t want_off[5] = {0, 1, 3, 3, 6};
    const int32_t want_perm[6] = {3, 1, 4, 0, 2, 5};
    int32_t off[5], perm[6];
    moe_host_cache* c = NULL;
    moe_expert_store* st = NULL;
    int hits = 0, i;

    CHECK(argc > 1);
    CHECK(strcmp(moe_status_str(MOE_OK), "MOE_OK") == 0);
    CHECK(strcmp(moe_status_str(MOE_EIO), "MOE_EIO") == 0);
    CHECK(strcmp(moe_status_str(MOE_EBUSY), "MOE_EBUSY") == 0);
    /* 27 * I * d / 16 bytes per expert; 221,184 is a multiple of 4096 */
    CHECK(moe_expert_bytes(&tiny) == 221184);
    CHECK(moe_store_expert_stride(&tiny) == 221184);

    /* the 3-slot LFU toy trace, one expert per step: 2 hits in 7 lookups */
    CHECK(moe_host_cache_create(16, 3, 0, &c) == MOE_OK);
    for (i = 0; i < 7; ++i) {
        int32_t slot, me[1], ms[1], nm, nh, nb;
        CHECK(moe_host_cache_step(c, &toy[i], 1, &slot, me, ms, &nm, &nh, &nb) == MOE_OK);
        CHECK(nm + nh == 1 && nb == 0 && slot >= 0 && slot < 3);
        hits += nh;
    }
    CHECK(hits == 2);
    moe_host_cache_destroy(c);

    /* stable grouping by expert */
    CHECK(moe_group_pairs(pair_ids, 6, 4, off, perm) == MOE_OK);
    CHECK(memcmp(off, want_off, sizeof off) == 0);
    CHECK(memcmp(perm, want_perm, sizeof perm) == 0);

    /* errors come back as status codes with a message */
    c = NULL;
    CHECK(moe_host_cache_create(0, 3, 0, &c) == MOE_EINVAL && c == NULL);
    CHECK(strlen(moe_last_error()) > 0);
    CHECK(moe_store_open(argv[1], &tiny, 2, 1, 0, &st) == MOE_EIO && st == NULL);
    CHECK(moe_store_open(argv[1], &tiny, 0, 1, 0, &st) == MOE_EINVAL);
    CHECK(moe_store_close(NULL) == MOE_OK);
    printf("abi ok\n");
    return 0;
}
