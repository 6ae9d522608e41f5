// placeholder: filled in with the tcgen05 kernel
#include "ct_internal.h"
namespace ct {
bool umma_supported(const Problem &, const Args *) { return false; }
size_t umma_workspace_bytes(const Problem &) { return 0; }
cudaError_t launch_umma(const Problem &, const Args &) { return cudaErrorNotSupported; }
}
