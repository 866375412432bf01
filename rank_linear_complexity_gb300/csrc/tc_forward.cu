// Tensor-core (tcgen05 / TMA) path: not wired yet.
#include "internal.cuh"

namespace linformer {

bool tc_supported(int, int, int, int) { return false; }

int tc_forward(const Problem &, float *, float *) { return LINFORMER_ERR_UNSUPPORTED; }

}  // namespace linformer
