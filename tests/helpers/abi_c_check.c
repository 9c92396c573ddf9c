/* A C11 caller of the library: compiles against include/h3fp4.h with a C
 * compiler (no C++), links libh3fp4.so, and checks entry points that need no
 * GPU (status strings, build information, host-side argument checks that
 * fail before anything is enqueued).  Prints "ok" and exits 0 on success. */
#include <stdio.h>
#include <string.h>

#include "h3fp4.h"

static int fail(const char *what)
{
    printf("FAILED: %s\n", what);
    return 1;
}

int main(void)
{
    const uintptr_t fake = 0x10000; /* 16-byte aligned; never dereferenced (every call below fails its checks) */
    void *d = (void *)fake;
    const int32_t offs[2] = {0, 10};
    h3fp4_gemm_config cfg;

    if (strcmp(h3fp4_status_string(H3FP4_OK), "ok") != 0)
        return fail("status string of H3FP4_OK");
    if (strstr(h3fp4_build_info(), "sm_103a") == NULL)
        return fail("build info names the target");
    /* producer: NULL tensor-scale output */
    if (h3fp4_modulate_absmax(d, 256, 10, 256, d, d, 256, offs, 1, NULL, (uint32_t *)d, NULL) != H3FP4_ERR_NULL)
        return fail("modulate_absmax rejects a NULL tensor scale");
    /* producer: m_pad not a multiple of 16 */
    if (h3fp4_modulate_pack(d, 256, 10, 24, 256, d, d, 256, offs, 1, (const float *)d, (uint8_t *)d, (uint8_t *)d,
                            NULL) != H3FP4_ERR_SHAPE)
        return fail("modulate_pack rejects m_pad % 16 != 0");
    /* GEMM: k not a multiple of 256, then an unknown kernel choice */
    if (h3fp4_gemm((const uint8_t *)d, (const uint8_t *)d, (const float *)d, (const uint8_t *)d, (const uint8_t *)d,
                   (const float *)d, d, 384, 300, 320, 384, 128, NULL, NULL) != H3FP4_ERR_SHAPE)
        return fail("gemm rejects k % 256 != 0");
    memset(&cfg, 0, sizeof cfg);
    cfg.cta_pair = 3;
    if (h3fp4_gemm((const uint8_t *)d, (const uint8_t *)d, (const float *)d, (const uint8_t *)d, (const uint8_t *)d,
                   (const float *)d, d, 384, 300, 320, 384, 256, &cfg, NULL) != H3FP4_ERR_UNSUPPORTED)
        return fail("gemm rejects an unknown kernel");
    if (h3fp4_device_error(NULL) != H3FP4_ERR_NULL)
        return fail("device_error rejects a NULL output");
    printf("ok\n");
    return 0;
}
