// Mask elements of the fused attention kernels, held packed between their
// load and their use: a boolean mask (MK = 2) four bytes per word, an
// additive 16-bit mask of the dtype T (MK = 1) two elements per word; no
// mask (MK = 0) one unused word.  32 elements (one chunk) per word array.
#pragma once

#include <stdint.h>

#include "sms_common.cuh"

namespace sms {

template <int MK> struct MaskWords { static constexpr int n = MK == 2 ? 8 : (MK == 1 ? 16 : 1); };

// Element e of a packed chunk as a log2-scaled score term: the additive value
// times log2(e), or 0 (kept) / -inf (masked) for a byte.
template <typename T, int MK>
__device__ __forceinline__ void mask_terms(const uint32_t (&w)[MaskWords<MK>::n], float (&m2)[32])
{
#pragma unroll
    for (int e = 0; e < 32; ++e) {
        if constexpr (MK == 1) {
            const uint16_t h = (uint16_t)(w[e >> 1] >> (16 * (e & 1)));
            m2[e] = to_f32<T>(*reinterpret_cast<const T *>(&h)) * kLog2e;
        } else if constexpr (MK == 2) {
            m2[e] = ((w[e >> 2] >> (8 * (e & 3))) & 0xffu) ? neg_inf() : 0.f;
        } else {
            m2[e] = 0.f;
        }
    }
}

// True when no element of the chunk, in any lane of the warp, is masked (all
// words zero: byte 0 = kept, additive +0).  Called by whole warps.
template <int MK> __device__ __forceinline__ bool mask_none(const uint32_t (&w)[MaskWords<MK>::n])
{
    uint32_t o = 0u;
#pragma unroll
    for (int k = 0; k < MaskWords<MK>::n; ++k) o |= w[k];
    return __all_sync(0xffffffffu, o == 0u);
}

}  // namespace sms
