// Host build of the library's exp_fast_f32 (csrc/moe_common.cuh) for
// tests/test_exp_fast_host.py: compiled with -ffp-contract=off, so every
// binary32 operation is rounded on its own as on the device.
#include "moe_common.cuh"

extern "C" void exp_fast_host_batch(const float* x, float* y, unsigned char* ok, long long n) {
  for (long long i = 0; i < n; ++i) {
    float v = 0.0f;
    ok[i] = moe::exp_fast_f32(x[i], &v) ? 1 : 0;
    y[i] = v;
  }
}
