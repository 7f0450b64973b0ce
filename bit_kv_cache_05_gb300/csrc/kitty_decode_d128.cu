// Kitty fused decode, D = 128: the instances for 1 ... 8 query heads per kv
// head (a translation unit of their own, compiled in parallel).
#include "kitty_decode.cuh"

namespace vqk {
namespace kitdec {

KitKernel pick_d128(int gq) { return pick<128>(gq); }

}  // namespace kitdec
}  // namespace vqk
