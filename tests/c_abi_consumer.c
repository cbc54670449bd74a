/*
 * A plain C program against include/kda.h and libkda.so, with no Python and no
 * CUDA headers: it checks the host-side parts of the C ABI that run without a
 * GPU (version, gate scale, launch plan, argument validation and the error
 * text). Built and run by tests/test_boundary_host.py; prints one line per
 * check and returns non-zero on the first failure.
 */
#include <math.h>
#include <stdio.h>
#include <string.h>

#include "kda.h"

#define CHECK(cond, what)                                  \
    do {                                                   \
        if (!(cond)) {                                     \
            printf("FAIL %s\n", what);                     \
            return 1;                                      \
        }                                                  \
        printf("ok %s\n", what);                           \
    } while (0)

int main(void)
{
    CHECK(kda_version() > 0, "version");
    CHECK(fabsf(kda_gate_scale(-5.0f) - (float)(-5.0 * 1.4426950408889634)) == 0.0f, "gate scale");

    int vs = 0;
    int64_t grid = 0;
    CHECK(kda_plan(128, 152, &vs, &grid) == KDA_OK && vs == 1 && grid == 128, "plan: one CTA per state");
    CHECK(kda_plan(32, 152, &vs, &grid) == KDA_OK && vs == 4 && grid == 128, "plan: V rows split four ways");
    CHECK(kda_plan(32, 152, NULL, &grid) == KDA_ERR_NULL, "plan: NULL output");

    /* dummy, never dereferenced, 16-byte aligned device addresses: every call below is rejected
       on the host before anything is launched */
    const void *q = (const void *)0x1000, *k = (const void *)0x2000, *v = (const void *)0x3000;
    const void *g = (const void *)0x4000, *beta = (const void *)0x5000;
    void *out = (void *)0x6000;
    kda_status st = kda_fwd(q, k, v, g, beta, 1.0f, out, NULL, NULL, -5.0f, NULL, KDA_DTYPE_NONE, NULL,
                            KDA_DTYPE_NONE, NULL, 0, 1, 16, 1, 64, 128, NULL);
    CHECK(st == KDA_ERR_SHAPE && strlen(kda_last_error()) > 0, "kda_fwd rejects K = 64");
    st = kda_fwd(q, k, v, g, beta, 1.0f, out, NULL, NULL, 0.5f, NULL, KDA_DTYPE_NONE, NULL, KDA_DTYPE_NONE,
                 NULL, 0, 1, 16, 1, 128, 128, NULL);
    CHECK(st == KDA_ERR_RANGE, "kda_fwd rejects lower_bound 0.5");
    st = kda_fwd_ex(q, k, v, g, beta, 1.0f, out, NULL, NULL, -5.0f, NULL, KDA_DTYPE_NONE, NULL, KDA_DTYPE_NONE,
                    NULL, 0, 1, 16, 1, 128, 128, 0x8u, NULL);
    CHECK(st == KDA_ERR_RANGE, "kda_fwd_ex rejects unknown option bits");

    kda_fwd_args a;
    memset(&a, 0, sizeof a);
    a.q = q; a.k = k; a.v = v; a.g = g; a.beta = beta; a.out = out;
    a.scale = 1.0f; a.lower_bound = -5.0f;
    a.B = 1; a.T = 16; a.H = 1; a.K = 128; a.V = 96;
    a.flags = KDA_FLAG_QK_L2NORM;
    CHECK(kda_fwd_packed(&a, NULL) == KDA_ERR_SHAPE, "kda_fwd_packed rejects V = 96");
    CHECK(kda_fwd_packed(NULL, NULL) == KDA_ERR_NULL, "kda_fwd_packed rejects a NULL struct");
    CHECK(kda_decode(q, k, v, g, beta, 1.0f, out, NULL, NULL, -5.0f, NULL, KDA_DTYPE_FP32, 2, 3, 128, 128,
                     NULL) == KDA_ERR_NULL,
          "kda_decode rejects a NULL state");
    return 0;
}
