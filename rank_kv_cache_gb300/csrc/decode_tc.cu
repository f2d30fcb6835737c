// tcgen05 rebuild path for the RoPE mode (placeholder until the kernel lands).
#include "internal.h"

namespace palu {

bool tc_supported(const DecodeArgs&) { return false; }
int tc_tile_tokens() { return 128; }
cudaError_t launch_decode_tc(const DecodeArgs&, cudaStream_t) { return cudaErrorNotSupported; }

}  // namespace palu
