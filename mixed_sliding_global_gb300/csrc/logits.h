// logits.h -- host-side interface of the final-logit soft-cap and greedy argmax kernels.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace gemma {

// row_ctas > 0: each row is split over row_ctas CTAs (at most 16) that form one cluster and
// reduce the row's index among themselves; one launch, no workspace (ws_bytes 0).
// row_ctas == 0: one wave of `n_cta` CTAs covers the flattened [batch][vocab] logits in equal
// contiguous ranges (a CTA's range may cross row boundaries); each (row, CTA) piece leaves one
// 64-bit word in the workspace, `ws_bytes` = (batch + n_cta) words, and a second launch
// reduces each row's words.
struct LogitPlan {
    int n_cta;
    size_t ws_bytes;
    int row_ctas;
};
LogitPlan logit_plan(int batch, int vocab, int n_sm);
cudaError_t launch_logit_softcap_argmax(const void* logits, void* capped, int32_t* argmax,
                                        void* workspace, int batch, int vocab, int fp32,
                                        float softcap, const LogitPlan& pl, cudaStream_t st);

}  // namespace gemma
