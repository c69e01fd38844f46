/* A plain C program that uses the library only through include/gdn.h: the
 * boundary must be consumable without C++, CUDA headers or torch.  Runs on a
 * machine without a GPU: it exercises the host-side entry points (version,
 * status strings, workspace sizes) and argument validation, which return
 * before any device work. */
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include "gdn.h"

#define CHECK(cond)                                                        \
    do {                                                                   \
        if (!(cond)) {                                                     \
            fprintf(stderr, "check failed at line %d: %s\n", __LINE__, #cond); \
            return 1;                                                      \
        }                                                                  \
    } while (0)

int main(void)
{
    CHECK(gdn_version() >= 100);
    CHECK(strcmp(gdn_status_string(GDN_OK), "ok") == 0);
    CHECK(strlen(gdn_status_string(GDN_ERR_WORKSPACE)) > 0);
    const size_t err = (size_t)-1;
    size_t ws = gdn_frame_fwd_workspace_size(1, 20, 121, 880, 112);
    CHECK(ws != err && ws > (size_t)20 * 121 * 78848);
    CHECK(gdn_frame_fwd_ex_workspace_size(1, 20, 121, 880, 112, GDN_FWD_REVERSE) == ws);
    /* the token-ordered reading adds one 8 KB T_off image per 64-token sub-chunk */
    CHECK(gdn_frame_fwd_ex_workspace_size(1, 20, 121, 880, 112, GDN_FWD_PRODUCT | GDN_FWD_REVERSE) >=
          ws + (size_t)20 * 121 * 14 * 8192);
    CHECK(gdn_frame_fwd_ex_workspace_size(1, 20, 121, 880, 112, GDN_FWD_PRODUCT) ==
          gdn_frame_fwd_product_workspace_size(1, 20, 121, 880, 112));
    CHECK(gdn_frame_fwd_ex_workspace_size(1, 20, 121, 880, 112, GDN_FWD_FUSED) == ws);
    CHECK(gdn_frame_fwd_ex_workspace_size(1, 20, 121, 880, 112, GDN_FWD_FUSED | GDN_FWD_PRODUCT) == err);
    CHECK(gdn_frame_fwd_ex_workspace_size(1, 20, 121, 880, 112, 8u) == err);
    CHECK(gdn_frame_fwd_workspace_size(1, 1, 2, 8, 64) == err);
    CHECK(gdn_frame_step_workspace_size(1, 20, 880, 112) == 0);
    CHECK(gdn_frame_bwd_workspace_size(1, 20, 121, 880, 112) != err);
    CHECK(gdn_frame_bwd_workspace_size(1, 20, 121, 0, 112) == err);
    /* validation before any device work */
    CHECK(gdn_frame_fwd(NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL, -1, 1, 1, 1, 112, 0.f, NULL, 0, NULL) ==
          GDN_ERR_INVALID_ARG);
    CHECK(gdn_frame_fwd(NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL, 0, 4, 4, 4, 112, 0.f, NULL, 0, NULL) ==
          GDN_OK); /* empty batch: no-op */
    CHECK(gdn_frame_fwd(NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL, 1, 1, 2, 8, 64, 0.f, NULL, 0, NULL) ==
          GDN_ERR_UNSUPPORTED);
    void *fake = (void *)(uintptr_t)0x10000; /* never dereferenced: validation fails first */
    CHECK(gdn_frame_fwd(fake, fake, fake, fake, fake, NULL, fake, fake, 1, 1, 2, 8, 112, 0.f, NULL, 0, NULL) ==
          GDN_ERR_WORKSPACE);
    CHECK(gdn_frame_fwd_ex(fake, fake, fake, fake, fake, NULL, fake, fake, 1, 1, 2, 8, 112, 0.f, 8u, fake, ws,
                           NULL) == GDN_ERR_INVALID_ARG);
    printf("abi consumer ok\n");
    return 0;
}
