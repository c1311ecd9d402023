// nf4_gemm placeholder (tcgen05 kernel not built yet).
#pragma once

#include "common.cuh"

namespace nf4q {

inline nf4q_status gemm_launch(const nf4q_weight*, const ScaleView&, const CodeValues&,
                               const void*, int64_t, void*, cudaStream_t, int) {
  return NF4Q_ERR_UNSUPPORTED;
}

}  // namespace nf4q
