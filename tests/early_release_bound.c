/* Host restatement of the single-launch step's early-release bound (clip_certainly_one
 * in the CUDA library): an fp32 upper bound of the sum of squares, its square root and
 * the bound of the fp64 path's divisor, all rounded upwards, as the device does with its
 * _ru intrinsics.  Built by tests/test_early_release_bound.py, which checks the bound
 * against the oracle's clip coefficient; the constants come from the CUDA source. */
#include <fenv.h>
#include <math.h>

/* gcc honours the rounding mode with -frounding-math (the test compiles with it); the
 * volatile temporaries keep each operation inside its fesetround bracket */

int certainly_one(float u, float max_norm, float k1, float k2, float k3)
{
    const int old = fegetround();
    fesetround(FE_UPWARD);
    volatile float b = sqrtf(u);
    volatile float t1 = b * k1;
    volatile float t2 = t1 + k2;
    volatile float need = t2 * k3;
    fesetround(old);
    return max_norm >= need;
}

/* the fp32 value nearest above (or equal to) x >= 0 */
float round_up_f32(double x)
{
    const int old = fegetround();
    fesetround(FE_UPWARD);
    volatile double v = x;
    volatile float f = (float)v;
    fesetround(old);
    return f;
}
