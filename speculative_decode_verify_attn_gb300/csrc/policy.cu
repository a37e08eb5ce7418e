// Confidence-gated draft depths (host code, no device work).
// Source: "Width vs. Depth: Speculating on the Margin": speculation efficiency varies per
// sequence, and allocating draft depth unevenly by drafter confidence beats fixed depths; it
// needs ragged speculation, which the verify kernels take (a depth per sequence).
//
// Reading: sequence b's drafted positions are each accepted with probability c_b, independently.
// A depth D commits 1 + c + ... + c^D tokens in expectation, so one more drafted position gains
// c^(D+1), a gain that shrinks with D. Handing out verify rows one at a time to the largest gain
// (ties to the lower sequence index) maximises the expected committed tokens under a row budget.
#include <cmath>
#include <cstdint>

#include "vfy.h"

extern "C" VFY_API vfy_status vfy_gate_depths(const float* confidence, int num_seqs, int row_budget,
                                              int max_depth, int32_t* depths) {
  if (num_seqs < 0 || max_depth < 0 || (num_seqs > 0 && (confidence == nullptr || depths == nullptr)))
    return VFY_EINVAL;
  for (int b = 0; b < num_seqs; ++b) {
    const float c = confidence[b];
    if (!(c >= 0.f && c <= 1.f)) return VFY_EINVAL;    // NaN fails too
    depths[b] = 0;
  }
  long long rows = num_seqs;                             // one row each for the committed token
  while (rows < row_budget) {
    int best = -1;
    double gain = -1.0;
    for (int b = 0; b < num_seqs; ++b) {
      if (depths[b] >= max_depth) continue;
      const double g = std::pow(static_cast<double>(confidence[b]), depths[b] + 1);
      if (g > gain) {
        best = b;
        gain = g;
      }
    }
    if (best < 0) break;
    ++depths[best];
    ++rows;
  }
  return VFY_OK;
}
