/* Compiles include/mla.h as strict C99 and calls the library's host-only
 * paths (version, status strings, argument checks) from C.  No GPU needed. */
#include <stdio.h>
#include <string.h>

#include "mla.h"

int main(void) {
    int fails = 0;
    if (mla_version() < 101) {
        printf("version %d\n", mla_version());
        ++fails;
    }
    if (!mla_status_string(MLA_ERR_UNSUPPORTED) || !strstr(mla_status_string(MLA_ERR_INVALID_ARG), "invalid"))
        ++fails;
    if (mla_absorb_q(NULL, NULL, NULL, 1, 1, 128, 512, MLA_BF16, NULL) != MLA_ERR_INVALID_ARG) ++fails;
    if (mla_cache_append(NULL, NULL, NULL, NULL, NULL, NULL, NULL, 1, 64, 16, 8, 1, 64, 1, 1, 10000.0,
                         NULL, 0, MLA_FP32, NULL) != MLA_ERR_INVALID_ARG)
        ++fails;
    if (mla_out_proj_merged(NULL, NULL, NULL, 1, 1, 64, 128, NULL, 0, MLA_BF16, NULL) !=
        MLA_ERR_INVALID_ARG)
        ++fails;
    if (mla_decode_workspace_size(0, 1, 128, 512, MLA_BF16) != 0) ++fails;
    {   /* RoPE widths past 128 are refused before any device work (the
         * pointers are never touched: they only have to be aligned) */
        void* fake = (void*)(size_t)4096;
        const int32_t* ifake = (const int32_t*)fake;
        if (mla_cache_append(fake, fake, fake, ifake, ifake, ifake, fake, 1, 64, 16, 130, 1, 64, 1, 1,
                             10000.0, NULL, 0, MLA_FP32, NULL) != MLA_ERR_UNSUPPORTED)
            ++fails;
        if (mla_project_q(fake, fake, ifake, fake, fake, 1, 1, 32, 130, 64, 10000.0, NULL, 0, MLA_FP32,
                          NULL) != MLA_ERR_UNSUPPORTED)
            ++fails;
        /* odd RoPE widths have no pairs */
        if (mla_project_q(fake, fake, ifake, fake, fake, 1, 1, 32, 15, 64, 10000.0, NULL, 0, MLA_FP32,
                          NULL) != MLA_ERR_INVALID_ARG)
            ++fails;
    }
    printf(fails ? "FAIL %d\n" : "ok\n", fails);
    return fails != 0;
}
