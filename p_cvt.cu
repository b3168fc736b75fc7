#include <cstdint>
__global__ void k(uint32_t* o, float a, float b){
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(a), "f"(b));
  o[0]=r;
}
