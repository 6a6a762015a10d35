#include <stdint.h>
__global__ void k(uint32_t* o, const uint32_t* i) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f16x2 %0, %1;" : "=h"(r) : "r"(i[threadIdx.x]));
  o[threadIdx.x] = r;
}
