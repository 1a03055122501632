/*
 * A plain C client of the library (no Python, no torch): it compiles against
 * include/fa.h alone, links libfa_gb300.so, and calls the entry points that
 * need no GPU -- the version, the status strings, argument checks that fail
 * before any device call, and the backward's workspace size.  Prints one
 * line per check; exits 0 when all hold.
 */
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include "fa.h"

static int failures = 0;

static void check(int ok, const char *what)
{
    printf("%s %s\n", ok ? "ok" : "FAIL", what);
    if (!ok) ++failures;
}

int main(void)
{
    /* fake, 16-byte aligned device addresses: never dereferenced */
    const uintptr_t P = (uintptr_t)1 << 20;
    void *q = (void *)P, *k = (void *)(2 * P), *v = (void *)(3 * P), *o = (void *)(4 * P);
    float *lse = (float *)(5 * P);
    size_t bytes = 0;

    check(fa_version() >= 100, "fa_version");
    check(strcmp(fa_status_string(FA_OK), "unknown status") != 0, "fa_status_string(FA_OK)");
    check(strcmp(fa_status_string((fa_status)99), "unknown status") == 0, "fa_status_string(99)");
    check(fa_fwd(NULL, k, v, o, lse, 1, 1, 16, 64, 0, 0.125f, NULL) == FA_ERR_INVALID_ARG, "null q");
    check(fa_fwd(q, k, v, o, lse, 1, 1, 0, 64, 0, 0.125f, NULL) == FA_ERR_INVALID_ARG, "N = 0");
    check(fa_fwd(q, k, v, o, lse, 1, 1, 16, 100, 0, 0.125f, NULL) == FA_ERR_UNSUPPORTED, "d = 100");
    check(fa_fwd(q, k, v, q, lse, 1, 1, 16, 64, 0, 0.125f, NULL) == FA_ERR_INVALID_ARG, "o aliases q");
    check(fa_fwd(q, k, v, o, lse, 1, 1, 16, 64, 2, 0.125f, NULL) == FA_ERR_INVALID_ARG, "causal = 2");
    check(fa_bwd_workspace_bytes(2, 3, 100, 128, &bytes) == FA_OK && bytes == (size_t)2 * 3 * 128 * 130 * 4,
          "fa_bwd_workspace_bytes");
    return failures ? 1 : 0;
}
