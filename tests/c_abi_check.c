/* A C11 caller of the library's host-side entry points (no GPU needed): the
 * header compiles as C, the symbols link, and the argument checks answer as
 * include/fd.h documents.  Exit status 0 when every check holds. */
#include <stdio.h>
#include <string.h>

#include "fd.h"

static int failures = 0;

static void expect(int ok, const char *what)
{
    if (!ok) {
        fprintf(stderr, "FAILED: %s\n", what);
        ++failures;
    }
}

int main(void)
{
    static const fd_status all[] = {FD_OK, FD_ERR_INVALID_ARG, FD_ERR_UNSUPPORTED, FD_ERR_WORKSPACE_TOO_SMALL,
                                    FD_ERR_CUDA, FD_ERR_TIMEOUT, FD_ERR_DEVICE_INPUT};
    const int n = (int)(sizeof all / sizeof all[0]);
    for (int i = 0; i < n; ++i) {
        const char *s = fd_status_string(all[i]);
        expect(s != NULL && s[0] != '\0', "every status has a name");
        for (int j = 0; j < i; ++j)
            expect(strcmp(s, fd_status_string(all[j])) != 0, "status names are distinct");
    }
    expect(fd_version() > 0, "version");

    /* workspace sizes: host-only, 0 for shapes no call accepts */
    const size_t ws = fd_workspace_size(4, 32, 8, 128, 4096, 0);
    expect(ws > 0, "workspace for GQA-4");
    expect(ws == fd_workspace_size(4, 32, 8, 128, 1000000, 16), "workspace independent of lengths");
    expect(fd_workspace_size_q(4, 32, 8, 128, 4096, 0, 1) == ws, "q_len 1 is the plain size");
    expect(fd_workspace_size_q(4, 16, 2, 128, 4096, 0, 2) > 0, "16 query columns");
    expect(fd_workspace_size_q(4, 16, 2, 128, 4096, 0, 3) == 0, "24 query columns: none");
    expect(fd_workspace_size(1, 32, 5, 128, 4096, 0) == 0, "Hq not a multiple of Hkv");

    /* argument checks answer before any launch */
    _Alignas(256) char buf[64];
    const void *q = buf;
    float *o = (float *)(void *)buf;
    expect(fd_decode(NULL, q, q, NULL, NULL, 2, 8, 2, 128, 64, 0.1f, o, NULL, buf, 1u << 30, NULL, NULL) ==
               FD_ERR_INVALID_ARG,
           "null q");
    expect(fd_decode(q, q, q, NULL, NULL, 2, 8, 2, 96, 64, 0.1f, o, NULL, buf, 1u << 30, NULL, NULL) ==
               FD_ERR_UNSUPPORTED,
           "head_dim 96");
    expect(fd_decode(q, q, q, NULL, NULL, 2, 8, 2, 128, 64, 0.1f, o, NULL, buf, 16, NULL, NULL) ==
               FD_ERR_WORKSPACE_TOO_SMALL,
           "small workspace");
    expect(fd_decode(q, q, q, NULL, NULL, 0, 8, 2, 128, 64, 0.1f, o, NULL, buf, 1u << 30, NULL, NULL) == FD_OK,
           "empty batch");
    expect(fd_decode_paged(q, q, q, (const int32_t *)q, 4, (const int32_t *)q, NULL, 2, 8, 2, 128, 24, 8, 0.1f,
                           o, NULL, buf, 1u << 30, NULL, NULL) == FD_ERR_UNSUPPORTED,
           "page size 24");
    fd_options opts;
    memset(&opts, 0, sizeof opts);
    opts.q_len = 2;
    opts.flags = FD_FLAG_CUDA_CORES;   /* 16 columns need the tensor cores */
    expect(fd_decode(q, q, q, NULL, NULL, 2, 16, 2, 128, 64, 0.1f, o, NULL, buf, 1u << 30, &opts, NULL) ==
               FD_ERR_UNSUPPORTED,
           "16 columns on CUDA cores");

    /* sequence sharding: a partial needs its LSE; the range is checked */
    expect(fd_decode_partial(q, q, q, NULL, NULL, 2, 8, 2, 128, 64, 0, 100, 0.1f, o, NULL, buf, 1u << 30, NULL,
                             NULL) == FD_ERR_INVALID_ARG,
           "partial without LSE");
    expect(fd_decode_partial(q, q, q, NULL, NULL, 2, 8, 2, 128, 64, 50, 40, 0.1f, o, o, buf, 1u << 30, NULL,
                             NULL) == FD_ERR_INVALID_ARG,
           "range end before its begin");
    expect(fd_decode_partial(q, q, q, NULL, NULL, 0, 8, 2, 128, 64, 0, 100, 0.1f, o, o, buf, 1u << 30, NULL,
                             NULL) == FD_OK,
           "empty batch partial");
    expect(fd_decode_paged_partial(q, q, q, (const int32_t *)q, 4, NULL, NULL, 2, 8, 2, 128, 16, 8, 0, 64, 0.1f,
                                   o, o, buf, 1u << 30, NULL, NULL) == FD_ERR_INVALID_ARG,
           "paged partial without lengths");
    expect(fd_merge_partials((const float *)q, (const float *)q, 0, 4, 128, o, NULL, NULL) == FD_ERR_INVALID_ARG,
           "merge of no sets");
    expect(fd_merge_partials((const float *)q, (const float *)q, 2, 4, 96, o, NULL, NULL) == FD_ERR_UNSUPPORTED,
           "merge head_dim 96");
    expect(fd_merge_partials((const float *)q, (const float *)q, 2, 0, 128, o, NULL, NULL) == FD_OK,
           "merge of no rows");

    if (failures == 0)
        printf("C ABI checks passed\n");
    return failures == 0 ? 0 : 1;
}
