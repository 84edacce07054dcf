// Inverse-frequency tables for scaled RoPE (host code).
//
// The "llama3" rule, published with Llama 3.1 and used by Llama-3.2 models,
// stretches a model trained on L = original_max_position tokens to longer
// contexts by slowing only its slow-turning dimensions.  With the wavelength
// of dimension i, lambda_i = 2 pi / inv_freq_i:
//   lambda_i < L / high_freq_factor:  kept as it is;
//   lambda_i > L / low_freq_factor:   divided by factor;
//   otherwise blended linearly in L / lambda_i between the two, weight
//   s = (L / lambda_i - low_freq_factor) / (high_freq_factor - low_freq_factor)
//   on the kept value.
// The pages of the fused-kernel sources apply no scaling; this table feeds
// ftk_qk_rope_freq_fwd/bwd, the same kernels with a caller's table.
#include <cmath>

#include "ftk.h"

extern "C" FTK_API ftk_status ftk_rope_llama3_inv_freq(int32_t D, double theta, double factor,
                                                      double low_freq_factor,
                                                      double high_freq_factor,
                                                      double original_max_position,
                                                      double *inv_freq) {
  if (!inv_freq) return FTK_ERR_NULL;
  if (D < 2 || D % 2 != 0 || D > 512 || !(theta > 1.0) || !(factor >= 1.0) ||
      !(low_freq_factor > 0.0) || !(high_freq_factor > low_freq_factor) ||
      !(original_max_position > 0.0) || !std::isfinite(theta) || !std::isfinite(factor) ||
      !std::isfinite(high_freq_factor) || !std::isfinite(original_max_position))
    return FTK_ERR_SHAPE;
  const double two_pi = 6.283185307179586476925;
  const double fast_edge = original_max_position / high_freq_factor;  // wavelengths below: kept
  const double slow_edge = original_max_position / low_freq_factor;   // above: divided
  for (int32_t i = 0; i < D / 2; ++i) {
    const double base = std::pow(theta, -2.0 * (double)i / (double)D);
    const double wavelength = two_pi / base;
    double out;
    if (wavelength < fast_edge) {
      out = base;
    } else if (wavelength > slow_edge) {
      out = base / factor;
    } else {
      const double keep = (original_max_position / wavelength - low_freq_factor) /
                          (high_freq_factor - low_freq_factor);
      out = keep * base + (1.0 - keep) * (base / factor);
    }
    inv_freq[i] = out;
  }
  return FTK_OK;
}
