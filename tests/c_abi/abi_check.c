/*
 * abi_check.c -- the library's C ABI used from plain C (no C++, no torch):
 * include/pfa.h compiles as C, every call takes plain pointers and sizes,
 * and argument validation and the host-side schedule replay run without a
 * GPU.  Built and run by tests/test_abi.py; exit status 0 means every check
 * passed, otherwise the number of the failed check.
 */
#include <stdio.h>
#include <string.h>

#include "pfa.h"

#define CHECK(n, cond)                                                  \
    do {                                                                \
        if (!(cond)) {                                                  \
            fprintf(stderr, "abi_check: check %d failed: %s\n", n, #cond); \
            return n;                                                   \
        }                                                               \
    } while (0)

int main(void)
{
    /* fake, aligned, disjoint device pointers: validation fails before any use */
    const void *q = (const void *)0x10000, *k = (const void *)0x20000000,
               *v = (const void *)0x40000000;
    void *out = (void *)0x60000000;

    CHECK(1, (pfa_version() >> 16) == 1);
    CHECK(2, strncmp(pfa_status_string(PFA_ERR_SHAPE), "PFA_ERR_SHAPE", 13) == 0);
    CHECK(3, pfa_prefill_attention(q, k, v, out, 16, 0, 8, 2, 128, 0, 0.1f, 7, NULL) ==
                 PFA_ERR_DTYPE);
    CHECK(4, pfa_prefill_attention(q, k, v, out, 16, 0, 6, 4, 128, 0, 0.1f, PFA_BF16, NULL) ==
                 PFA_ERR_SHAPE);
    CHECK(5, pfa_prefill_attention(NULL, k, v, out, 16, 0, 8, 2, 128, 0, 0.1f, PFA_BF16, NULL) ==
                 PFA_ERR_NULL);
    CHECK(6, pfa_prefill_attention(q, k, v, out, 0, 0, 8, 2, 128, 0, 0.1f, PFA_BF16, NULL) ==
                 PFA_OK);
    CHECK(7, pfa_prefill_attention_cache(q, k, v, out, 16, 100, 8, 2, 128, 0, 0.1f, PFA_BF16,
                                         8 * 128, 512, 1, NULL, 0, NULL) == PFA_ERR_SHAPE);
    {
        int schedule = -1, ctas = -1, failed = -1;
        CHECK(8, pfa_debug_check_schedule(1358, 0, 32, 8, 0, 152, &schedule, &ctas, &failed) ==
                     PFA_OK);
        CHECK(9, schedule == PFA_SCHEDULE_PLAIN && ctas == 176 && failed == 0);
        CHECK(10, pfa_debug_check_schedule(2048, 61440, 32, 8, 0, 152, &schedule, &ctas,
                                           &failed) == PFA_OK);
        CHECK(11, schedule == PFA_SCHEDULE_TAIL && failed == 0);
        CHECK(16, pfa_debug_check_schedule_d512(2048, 6144, 8, 2, 1024, 152, &schedule, &ctas,
                                                &failed) == PFA_OK);
        CHECK(17, schedule == PFA_SCHEDULE_PLAIN && ctas == 256 && failed == 0);
    }
    {
        /* the host-buffer entry: checks that need no device */
        size_t bytes = 1;
        void *dbuf = (void *)0x7000000000;
        CHECK(12, pfa_host_buffer_bytes(16, 0, 6, 4, 128, 0, PFA_BF16, &bytes) == PFA_ERR_SHAPE);
        CHECK(13, pfa_host_buffer_bytes(0, 0, 8, 2, 128, 0, PFA_BF16, &bytes) == PFA_OK &&
                      bytes == 0);
        CHECK(14, pfa_prefill_attention_host(q, k, v, out, 16, 0, 8, 2, 128, 0, 0.1f, PFA_BF16,
                                             NULL, 1 << 20, NULL) == PFA_ERR_NULL);
        CHECK(15, pfa_prefill_attention_host(q, k, v, out, 16, 0, 8, 2, 128, 0, 0.1f, PFA_BF16,
                                             (char *)dbuf + 16, 1 << 20, NULL) ==
                      PFA_ERR_ALIGNMENT);
    }
    printf("abi_check: all checks passed\n");
    return 0;
}
