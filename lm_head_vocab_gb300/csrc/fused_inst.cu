// Instantiations of the staged-row kernel for one (dtype, teacher, temperature,
// entropy) combination, chosen by LMLOSS_FUSED_VARIANT (0..7) when this file
// is compiled; the library links the eight objects.
#include "kernels.cuh"
#include "fused_entry.cuh"

#ifndef LMLOSS_FUSED_VARIANT
#error "compile with -DLMLOSS_FUSED_VARIANT=0..7"
#endif

namespace lmloss {

template <bool BF16, bool KL, bool TAU, bool ENT>
const void* fused_entry(int nt, bool stats)
{
    switch (nt) {
    case 128:
        return stats ? reinterpret_cast<const void*>(&fused_kernel<BF16, KL, 128, true, TAU, ENT>)
                     : reinterpret_cast<const void*>(&fused_kernel<BF16, KL, 128, false, TAU, ENT>);
    case 256:
        return stats ? reinterpret_cast<const void*>(&fused_kernel<BF16, KL, 256, true, TAU, ENT>)
                     : reinterpret_cast<const void*>(&fused_kernel<BF16, KL, 256, false, TAU, ENT>);
    case 512:
        return stats ? reinterpret_cast<const void*>(&fused_kernel<BF16, KL, 512, true, TAU, ENT>)
                     : reinterpret_cast<const void*>(&fused_kernel<BF16, KL, 512, false, TAU, ENT>);
    case 1024:
        return stats ? reinterpret_cast<const void*>(&fused_kernel<BF16, KL, 1024, true, TAU, ENT>)
                     : reinterpret_cast<const void*>(&fused_kernel<BF16, KL, 1024, false, TAU, ENT>);
    default:
        return nullptr;
    }
}

// variants 0..5: 3 * (fp32) + (0 plain, 1 teacher, 2 teacher at a temperature);
// 6, 7: plain with the entropy, bf16 and fp32
#define LMLOSS_V LMLOSS_FUSED_VARIANT
#if LMLOSS_V < 0 || LMLOSS_V > 7
#error "LMLOSS_FUSED_VARIANT must be 0..7"
#endif
#if LMLOSS_V < 6
template const void* fused_entry<(LMLOSS_V < 3), (LMLOSS_V % 3) != 0, (LMLOSS_V % 3) == 2, false>(int, bool);
#else
template const void* fused_entry<(LMLOSS_V == 6), false, false, true>(int, bool);
#endif
#undef LMLOSS_V

}  // namespace lmloss
