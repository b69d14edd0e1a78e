// Addresses of the staged-row kernel's instantiations.  Each (dtype, teacher,
// temperature, entropy) combination built is instantiated in its own object file,
// compiled from fused_inst.cu, so that the library's translation units build
// in parallel; the host code reaches them only through these functions.
#pragma once

namespace lmloss {

// fused_kernel<BF16, KL, nt, stats, TAU, ENT> for a block of nt threads (128,
// 256, 512 or 1024), or null for any other nt.  stats selects the
// statistics-pass instantiation (no gradient, early buffer hand-off).
template <bool BF16, bool KL, bool TAU, bool ENT>
const void* fused_entry(int nt, bool stats);

extern template const void* fused_entry<true, false, false, false>(int, bool);
extern template const void* fused_entry<true, true, false, false>(int, bool);
extern template const void* fused_entry<true, true, true, false>(int, bool);
extern template const void* fused_entry<false, false, false, false>(int, bool);
extern template const void* fused_entry<false, true, false, false>(int, bool);
extern template const void* fused_entry<false, true, true, false>(int, bool);
// the entropy as a compile-time choice exists without a teacher only
extern template const void* fused_entry<true, false, false, true>(int, bool);
extern template const void* fused_entry<false, false, false, true>(int, bool);

}  // namespace lmloss
