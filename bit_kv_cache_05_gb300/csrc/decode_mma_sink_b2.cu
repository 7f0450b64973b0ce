// Instantiations of the tensor-core decode kernel for 2-bit KIVI-Sink caches
// (sink tokens' quantized scores masked): D in
// {64, 128}, 1/2/4 query heads per kv head (padded), group size 16..128.
#include "decode_mma.cuh"

namespace vqk {
namespace mma {

bool kernel_sink_b2(int D, int GQP, int G, KernelInfo *out) {
#define VQK_CASE(DD, QQ, GG)                                   \
  if (D == DD && GQP == QQ && G == GG) {                       \
    *out = info<Cfg<DD, 2, QQ, GG, true>>();                        \
    return true;                                               \
  }
#define VQK_ALL_G64(QQ) VQK_CASE(64, QQ, 16) VQK_CASE(64, QQ, 32) VQK_CASE(64, QQ, 64)
#define VQK_ALL_G128(QQ) \
  VQK_CASE(128, QQ, 16) VQK_CASE(128, QQ, 32) VQK_CASE(128, QQ, 64) VQK_CASE(128, QQ, 128)
  VQK_ALL_G64(1) VQK_ALL_G64(2) VQK_ALL_G64(4)
  VQK_ALL_G128(1) VQK_ALL_G128(2) VQK_ALL_G128(4)
#undef VQK_ALL_G128
#undef VQK_ALL_G64
#undef VQK_CASE
  return false;
}

}  // namespace mma
}  // namespace vqk
