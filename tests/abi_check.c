/* Plain-C client of libfp4q.so: the public header compiles as C99 and the
 * library links and answers from C alone.  Only host-side paths run (status
 * strings and argument validation), so no GPU is needed. */
#include <stdio.h>
#include <string.h>

#include "fp4q.h"

int main(void) {
    int fails = 0;
    for (int s = FP4Q_OK; s <= FP4Q_ERR_TIMEOUT; ++s) {
        const char* msg = fp4q_status_string((fp4q_status)s);
        if (!msg || !msg[0]) { printf("empty status string %d\n", s); ++fails; }
    }
    /* validation happens before any device work */
    if (fp4q_quantize(NULL, 17, 16, FP4Q_AXIS_ROW, FP4Q_SCALE_UE5M3, NULL, FP4Q_RNE, 0,
                      NULL, NULL, NULL, NULL, NULL, NULL, NULL) == FP4Q_OK) ++fails;
    if (fp4q_gemm(NULL, NULL, NULL, NULL, NULL, NULL, 128, 128, 96, FP4Q_SCALE_UE5M3,
                  NULL, 0, NULL) != FP4Q_ERR_SHAPE) ++fails;
    if (fp4q_amax(NULL, 16, NULL, NULL) != FP4Q_ERR_ARG) ++fails;
    if (fp4q_get_device_status(NULL, NULL) != FP4Q_ERR_ARG) ++fails;
    printf(fails ? "FAIL %d\n" : "ok\n", fails);
    return fails != 0;
}
