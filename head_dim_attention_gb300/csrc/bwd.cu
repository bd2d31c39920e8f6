// Attention backward: not yet implemented in this revision of the library.
#include "internal.h"
namespace ffpa {
cudaError_t launch_bwd(const BwdParams&, const BwdMaps&, bool, cudaStream_t) { return cudaErrorNotSupported; }
}  // namespace ffpa
