/*
 * Plain C client of the bstq C ABI (no Python, no torch): includes bstq.h,
 * links libbstq.so and makes the calls that need no GPU: version, status
 * text, argument validation and, where no device is visible, the
 * no-device status.  Built and run by tests/test_c_client.py.
 * Prints one line per check; exits non-zero on the first mismatch.
 */
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include "bstq.h"

static int fails = 0;

static void expect(const char *what, int got, int want)
{
    printf("%s: %d (want %d)\n", what, got, want);
    if (got != want)
        ++fails;
}

int main(int argc, char **argv)
{
    const int have_gpu = argc > 1 && strcmp(argv[1], "gpu") == 0;
    static double buf[64];
    void *p = buf;
    const char *v = bstq_version();
    printf("version: %s\n", v);
    if (strncmp(v, "bstq", 4) != 0)
        ++fails;
    if (strcmp(bstq_status_string(0), "success") != 0)
        ++fails;

    expect("solve dtype", bstq_solve((bstq_dtype)7, BSTQ_JOBZ_V, 8, 10, p, p, p, p, NULL), -1);
    expect("solve jobz", bstq_solve(BSTQ_F32, (bstq_jobz)5, 8, 10, p, p, p, p, NULL), -2);
    expect("solve n", bstq_solve(BSTQ_F32, BSTQ_JOBZ_V, BSTQ_MAX_N + 1, 10, p, p, p, p, NULL), -3);
    expect("solve batch", bstq_solve(BSTQ_F32, BSTQ_JOBZ_V, 8, -1, p, p, p, p, NULL), -4);
    expect("solve empty batch", bstq_solve(BSTQ_F32, BSTQ_JOBZ_V, 8, 0, NULL, NULL, NULL, NULL, NULL), 0);
    expect("solve d", bstq_solve(BSTQ_F64, BSTQ_JOBZ_V, 8, 10, NULL, p, p, p, NULL), -5);
    expect("solve e", bstq_solve(BSTQ_F64, BSTQ_JOBZ_V, 8, 10, p, NULL, p, p, NULL), -6);
    expect("solve Q", bstq_solve(BSTQ_F64, BSTQ_JOBZ_V, 8, 10, p, p, NULL, p, NULL), -7);
    expect("solve work", bstq_solve(BSTQ_F64, BSTQ_JOBZ_V, 8, 10, p, p, p, NULL, NULL), -8);

    bstq_params prm;
    memset(&prm, 0, sizeof(prm));
    prm.scheduler = 9;
    expect("solve_ex params", bstq_solve_ex(BSTQ_F32, BSTQ_JOBZ_V, 8, 10, p, p, p, p, NULL, &prm), -10);
    memset(&prm, 0, sizeof(prm));
    prm.log_entries = -1;
    expect("solve_ex log entries", bstq_solve_ex(BSTQ_F32, BSTQ_JOBZ_V, 64, 10, p, p, p, p, NULL, &prm), -10);

    expect("stedc_leaves leaf", bstq_stedc_leaves(BSTQ_F32, BSTQ_JOBZ_V, 70, 0, 10, p, p, p, (int32_t *)p, p,
                                                  NULL, NULL), -3);
    expect("syev n", bstq_syev(BSTQ_F32, BSTQ_JOBZ_V, 40, 10, p, p, p, p, NULL, NULL), -3);

    if (!have_gpu) {
        /* valid arguments: the library must say that no device is usable */
        expect("solve without a device", bstq_solve(BSTQ_F32, BSTQ_JOBZ_V, 8, 10, p, p, p, p, NULL),
               BSTQ_ERR_NODEVICE);
        expect("work size without a device", (int)bstq_work_size(BSTQ_F32, BSTQ_JOBZ_V, 8, 10), 0);
    }
    printf("%s\n", fails ? "FAIL" : "OK");
    return fails ? 1 : 0;
}
