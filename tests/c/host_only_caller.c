/*
 * A caller of libnts written in plain C, with host buffers only: it reads
 * bf16 rows from a file, runs MXNorm (p = 2) + E4M3 cast through
 * nts_mxnorm_cast_host_noalloc (the library stages the rows in its own
 * device array: this program allocates no device memory and includes no
 * CUDA header), and writes the codes and then the scales to a file.
 *
 *   host_only_caller --checks                 argument checks only (no GPU)
 *   host_only_caller IN OUT T D               IN: T*D bf16 values (uint16)
 *
 * Exit status 0 on success; otherwise the library's status is printed.
 */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "nts.h"

static int expect(int got, int want, const char *what) {
    if (got == want) return 0;
    fprintf(stderr, "%s: got %s, want %s (%s)\n", what, nts_status_string(got),
            nts_status_string(want), nts_last_error());
    return 1;
}

static int checks(void) {
    static uint16_t x[4 * 64];
    static uint8_t codes[4 * 64], scales[4 * 2];
    double c = 0.0;
    int bad = 0;
    if (nts_version() < 100) bad = 1;
    bad |= expect(nts_mxnorm_cast_host_noalloc(NULL, NULL, codes, scales, 4, 64, 1e-6f, 32,
                                               NTS_FMT_E4M3, 2, NULL),
                  NTS_ERR_INVALID_ARG, "NULL input");
    bad |= expect(nts_mxnorm_cast_host_noalloc(x, NULL, codes, scales, 4, 64, 1e-6f, 8,
                                               NTS_FMT_E4M3, 2, NULL),
                  NTS_ERR_INVALID_ARG, "block size 8");
    bad |= expect(nts_mxnorm_cast_host_noalloc(x, NULL, codes, scales, 0, 64, 1e-6f, 32,
                                               NTS_FMT_E4M3, 2, NULL),
                  NTS_OK, "no tokens");
    bad |= expect(nts_mxnorm_correction(32, 2, &c), NTS_OK, "c(32, 2)");
    if (c < 0.418 || c > 0.419) {
        fprintf(stderr, "c(32, 2) = %.10f\n", c);
        bad = 1;
    }
    return bad;
}

int main(int argc, char **argv) {
    if (argc == 2 && strcmp(argv[1], "--checks") == 0) return checks();
    if (argc != 5) {
        fprintf(stderr, "usage: %s --checks | IN OUT T D\n", argv[0]);
        return 2;
    }
    const long T = atol(argv[3]), D = atol(argv[4]), B = 32;
    uint16_t *x = malloc((size_t)T * D * 2);
    uint8_t *codes = malloc((size_t)T * D);
    uint8_t *scales = malloc((size_t)T * (D / B));
    FILE *f = fopen(argv[1], "rb");
    if (!x || !codes || !scales || !f || fread(x, 2, (size_t)T * D, f) != (size_t)T * D) {
        fprintf(stderr, "cannot read %s\n", argv[1]);
        return 2;
    }
    fclose(f);
    int rc = nts_mxnorm_cast_host_noalloc(x, NULL, codes, scales, T, D, 1e-6f, (int)B,
                                          NTS_FMT_E4M3, 2, NULL);
    if (rc == NTS_OK) rc = nts_check_status(NULL);
    if (rc != NTS_OK) {
        fprintf(stderr, "libnts: %s: %s\n", nts_status_string(rc), nts_last_error());
        return 1;
    }
    f = fopen(argv[2], "wb");
    if (!f || fwrite(codes, 1, (size_t)T * D, f) != (size_t)T * D ||
        fwrite(scales, 1, (size_t)T * (D / B), f) != (size_t)T * (D / B)) {
        fprintf(stderr, "cannot write %s\n", argv[2]);
        return 2;
    }
    fclose(f);
    free(x);
    free(codes);
    free(scales);
    return 0;
}
