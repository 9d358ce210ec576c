// K2: tcgen05 attention forward (placeholder until the kernel lands).
#include "common.cuh"
#include "internal.h"

namespace ulysses {
ULYSSES_ERROR_READER(read_error_attn_tc_fwd)
bool tc_fwd_supported(const AttnArgs&) { return false; }
int launch_tc_fwd(const AttnArgs&, cudaStream_t) {
  return set_error(ULYSSES_ERR_UNSUPPORTED, "tcgen05 forward not built");
}
}  // namespace ulysses
