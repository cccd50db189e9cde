// decode_util.cuh -- helpers shared by the CUDA-core paged decode kernels.
#pragma once

#include <cstdint>

namespace fattn {

// The first nv of the eight 16-bit values in v (memory order), the others
// cleared to +0.  Used on cache slots past a sequence's context, whose bits are
// arbitrary: a zero attention weight does not cancel a NaN or an infinity.
__device__ __forceinline__ uint4 keep_first_16b(uint4 v, int nv) {
  auto k2 = [nv](uint32_t w, int i) -> uint32_t {
    return i + 1 < nv ? w : (i < nv ? (w & 0xffffu) : 0u);
  };
  return make_uint4(k2(v.x, 0), k2(v.y, 2), k2(v.z, 4), k2(v.w, 6));
}

}  // namespace fattn
