/*
 * A plain C99 caller of libmamba2.so: include/mamba2.h must compile as C and
 * every call below must link and return what the header promises on a host
 * without a GPU (only argument checks and queries run; nothing is launched).
 * Prints one line per failed check and exits with the number of failures.
 */
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include "mamba2.h"

static int failures = 0;

#define CHECK(cond)                                                     \
    do {                                                                \
        if (!(cond)) {                                                  \
            printf("FAILED line %d: %s\n", __LINE__, #cond);            \
            ++failures;                                                 \
        }                                                               \
    } while (0)

/* distinct, 16-byte aligned addresses that are never dereferenced on the host */
static void* fake(int i) { return (void*)(uintptr_t)(0x100000u + 256u * (unsigned)i); }

int main(void) {
    /* the Nemotron-H mixer shape, bf16 activations */
    m2_dims d;
    memset(&d, 0, sizeof d);
    d.batch = 1;
    d.T = 300;
    d.nheads = 128;
    d.headdim = 80;
    d.dstate = 128;
    d.ngroups = 8;
    d.dconv = 4;
    d.act = M2_BF16;

    /* status strings: one for every code, and a fallback */
    for (int s = M2_OK; s <= M2_EWORKSPACE; ++s) {
        const char* str = mamba2_status_string((m2_status)s);
        CHECK(str != NULL && str[0] != '\0');
    }
    CHECK(strcmp(mamba2_status_string((m2_status)99), "unknown status") == 0);

    /* workspace queries */
    CHECK(mamba2_scan_workspace_bytes(&d, 128) > 0);
    CHECK(mamba2_scan_workspace_bytes(&d, 0) == 0);
    CHECK(mamba2_scan_workspace_bytes(NULL, 128) == 0);
    const size_t ws_step = mamba2_step_workspace_bytes(&d, 64);
    CHECK(ws_step >= (size_t)64 * (12288 + 128) * 4);
    CHECK(mamba2_step_workspace_bytes(&d, -1) == 0);
    CHECK(mamba2_step_noalloc_max_bytes() == ((size_t)1 << 20));
    CHECK(mamba2_attn_decode_workspace_bytes(1, 40, 8, 128, 750, M2_BF16) == 0);
    CHECK(mamba2_attn_decode_workspace_bytes(1, 40, 8, 64, 750, M2_BF16) == 0);

    /* the step: a NULL input, a misaligned input, a short workspace, a bad shape */
    void* p[12];
    for (int i = 0; i < 12; ++i) p[i] = fake(i);
    CHECK(mamba2_step(&d, 2, NULL, p[1], p[2], p[3], (const float*)p[4], (const float*)p[5], (const float*)p[6],
                      (const float*)p[7], (const float*)p[8], (float*)p[9], p[10], p[11], fake(40), ws_step,
                      NULL) == M2_EINVAL);
    CHECK(mamba2_step(&d, 2, (char*)p[0] + 2, p[1], p[2], p[3], (const float*)p[4], (const float*)p[5],
                      (const float*)p[6], (const float*)p[7], (const float*)p[8], (float*)p[9], p[10], p[11],
                      fake(40), ws_step, NULL) == M2_EALIGN);
    CHECK(mamba2_step(&d, 64, p[0], p[1], p[2], p[3], (const float*)p[4], (const float*)p[5], (const float*)p[6],
                      (const float*)p[7], (const float*)p[8], (float*)p[9], p[10], p[11], fake(40), ws_step - 1,
                      NULL) == M2_EWORKSPACE);
    m2_dims bad = d;
    bad.dconv = 3;
    CHECK(mamba2_step(&bad, 2, p[0], p[1], p[2], p[3], (const float*)p[4], (const float*)p[5],
                      (const float*)p[6], (const float*)p[7], (const float*)p[8], (float*)p[9], p[10], p[11],
                      fake(40), ws_step, NULL) == M2_ESHAPE);
    CHECK(mamba2_step_noalloc(&d, 22, p[0], p[1], p[2], p[3], (const float*)p[4], (const float*)p[5],
                              (const float*)p[6], (const float*)p[7], (const float*)p[8], (float*)p[9], p[10],
                              p[11], NULL) == M2_EWORKSPACE);

    /* the scan: chunk out of range */
    CHECK(mamba2_conv_scan(&d, p[0], p[1], p[2], p[3], (const float*)p[4], (const float*)p[5], (const float*)p[6],
                           (const float*)p[7], (const float*)p[8], 129, NULL, NULL, p[9], (float*)p[10], p[11],
                           fake(40), (size_t)1 << 40, NULL) == M2_EINVAL);

    /* the 4-bit projection: only group 64, 4 bits; in_features a multiple of 64 */
    CHECK(mamba2_qlinear(300, 4480, 22656, 32, 4, p[0], (const uint32_t*)p[1], p[2], p[3], p[4], NULL) ==
          M2_EUNSUPPORTED);
    CHECK(mamba2_qlinear(300, 4481, 22656, 64, 4, p[0], (const uint32_t*)p[1], p[2], p[3], p[4], NULL) ==
          M2_ESHAPE);
    /* the fused form with a gated norm whose groups do not divide the row */
    m2_row_norm nm;
    memset(&nm, 0, sizeof nm);
    nm.kind = M2_NORM_GATED;
    nm.weight = (const float*)p[5];
    nm.eps = 1e-5f;
    nm.groups = 3;
    nm.gate = p[6];
    nm.gate_stride = 22656;
    CHECK(mamba2_qlinear_fused(300, 10240, 4480, 64, 4, p[0], 10240, &nm, (const uint32_t*)p[1], p[2], p[3],
                               NULL, p[4], NULL) == M2_ESHAPE);

    /* the language model: an unknown block kind; no description at all */
    m2_lm_layer layers[2];
    memset(layers, 0, sizeof layers);
    m2_lm m;
    memset(&m, 0, sizeof m);
    m.n_layers = 2;
    m.kinds = "MX";
    m.layers = layers;
    m.hidden = 4480;
    m.mixer = d;
    m.norm_eps = 1e-5f;
    CHECK(mamba2_lm_workspace_bytes(&m, 1, 1, 1) == 0);
    CHECK(mamba2_lm_step(&m, 1, fake(50), NULL, NULL, 0, NULL) == M2_EINVAL);
    CHECK(mamba2_lm_workspace_bytes(NULL, 1, 1, 1) == 0);
    m.kinds = "MM";
    CHECK(mamba2_lm_workspace_bytes(&m, 1, 300, 128) > 0);

    /* the device error word needs somewhere to put the code */
    CHECK(mamba2_device_error(NULL, NULL) == M2_EINVAL);

    printf("%s: %d failed\n", failures ? "FAILED" : "ok", failures);
    return failures;
}
