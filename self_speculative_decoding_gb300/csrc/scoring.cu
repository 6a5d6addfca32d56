// SWIFT §4.1.2 candidate-mask scoring (ssd_score_masks).
#include <string>

#include "../../include/ssd.h"

extern "C" ssd_status ssd_score_masks(ssd_ctx* ctx, const uint64_t* masks, int32_t K, int32_t N,
                                      float* matchness_out, int32_t* best_out) {
  (void)ctx; (void)masks; (void)K; (void)N; (void)matchness_out; (void)best_out;
  return SSD_ERR_INVALID_ARG;
}
