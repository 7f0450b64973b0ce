// Kitty fused decode, D = 64: the instances for 1 ... 8 query heads per kv
// head (a translation unit of their own, compiled in parallel).
#include "kitty_decode.cuh"

namespace vqk {
namespace kitdec {

KitKernel pick_d64(int gq) { return pick<64>(gq); }

}  // namespace kitdec
}  // namespace vqk
