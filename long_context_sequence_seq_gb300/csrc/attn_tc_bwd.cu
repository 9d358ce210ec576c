// K4: tcgen05 attention backward (placeholder until the kernel lands).
#include "common.cuh"
#include "internal.h"

namespace ulysses {
ULYSSES_ERROR_READER(read_error_attn_tc_bwd)
bool tc_bwd_supported(const AttnArgs&) { return false; }
int launch_tc_bwd(const AttnArgs&, cudaStream_t) {
  return set_error(ULYSSES_ERR_UNSUPPORTED, "tcgen05 backward not built");
}
}  // namespace ulysses
