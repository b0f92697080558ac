/*
 * A plain C99 caller of the library: includes the public header as C, links
 * the shared library, and calls entry points that need no device (version,
 * status text, host-side argument checks, zero-row calls). Exits 0 when every
 * check holds. Built and run by tests/test_abi_from_c.py.
 */
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include "ce_rows.h"

static int failures = 0;

static void expect(int cond, const char *what)
{
    if (!cond) {
        printf("FAILED: %s\n", what);
        ++failures;
    }
}

int main(void)
{
    expect(ce_version() == 10000, "version");
    expect(strlen(ce_status_string(CE_EINVAL)) > 0, "status text");
    /* argument checks run on the host before any device is touched */
    expect(ce_rows(NULL, 4, 10, 10, NULL, NULL, NULL) == CE_EINVAL, "ce_rows: null logits");
    expect(ce_grad((const float *)256, 4, 10, 9, (const int64_t *)512, 1.0, (float *)4096, NULL, NULL) == CE_EINVAL,
           "ce_grad: stride < vocab");
    expect(ce_loss((const float *)256, 4, 10, 10, (const int64_t *)512, (float *)1024, NULL, NULL) == CE_EINVAL,
           "ce_loss: no mean");
    expect(ce_grad_step((const float *)256, 4, 10, 10, (const int64_t *)512, 1.0, (float *)4096, NULL, NULL,
                        (double *)8192, NULL) == CE_EINVAL,
           "ce_grad_step: a mean without row losses");
    expect(argmax_rows((const float *)258, 4, 10, 10, (float *)1024, NULL) == CE_EALIGN,
           "argmax_rows: misaligned logits");
    expect(ce_device_error_count(NULL, NULL) == CE_EINVAL, "ce_device_error_count: no output");
    expect(ce_device_wait_timeouts(NULL, NULL) == CE_EINVAL, "ce_device_wait_timeouts: no output");
    expect(split_sum((float *)256, (const float *)4096, 10, 0, 0, NULL) == CE_EINVAL, "split_sum: no parts");
    expect(candidates_rows((const float *)256, 4, 0, 10, (float *)8192, NULL) == CE_EINVAL,
           "candidates_rows: vocab < 1");
    expect(argmax_rows_indirect(NULL, 4, 10, (float *)4096, NULL) == CE_EINVAL, "indirect: no table");
    /* zero rows: nothing to do, nothing launched */
    expect(ce_rows(NULL, 0, 10, 10, NULL, NULL, NULL) == CE_OK, "ce_rows: zero rows");
    expect(softmax_rows(NULL, 0, 10, 10, NULL, NULL) == CE_OK, "softmax_rows: zero rows");
    expect(argmax_rows(NULL, 0, 10, 10, NULL, NULL) == CE_OK, "argmax_rows: zero rows");
    expect(ce_grad(NULL, 0, 10, 10, NULL, 1.0, NULL, NULL, NULL) == CE_OK, "ce_grad: zero rows");
    expect(ce_debug_force(0, 0, 0) == CE_OK, "debug_force reset");
    expect(ce_debug_force(7, 2, 0) == CE_OK && ce_debug_force(0, 0, 0) == CE_OK, "debug_force: the ring path");
    expect(ce_debug_grid_cap(-1) == CE_EINVAL, "grid cap: negative");
    expect(ce_debug_grid_cap(0) == CE_OK, "grid cap: none");
    /* the host-fed step: argument checks answer before any copy */
    expect(ce_grad_host(NULL, 4, 10, 10, (const int64_t *)512, 1.0, (float *)4096, (int64_t *)8192,
                        (float *)16384, (float *)32768, NULL, (double *)65536, NULL, NULL, 0, NULL) == CE_EINVAL,
           "ce_grad_host: null host logits");
    expect(ce_grad_host((const float *)256, 4, 10, 10, (const int64_t *)516, 1.0, (float *)4096,
                        (int64_t *)8192, (float *)16384, (float *)32768, NULL, (double *)65536, NULL, NULL, 0,
                        NULL) == CE_EALIGN,
           "ce_grad_host: misaligned host labels");
    expect(ce_grad_host((const float *)256, 4, 10, 10, (const int64_t *)512, 1.0, (float *)4096,
                        (int64_t *)8192, (float *)16384, (float *)32768, NULL, (double *)65536, NULL,
                        (float *)1024, 0, NULL) == CE_EINVAL,
           "ce_grad_host: tokens back without device tokens");
    printf("%s\n", failures ? "abi from C: FAILED" : "abi from C: ok");
    return failures ? 1 : 0;
}
