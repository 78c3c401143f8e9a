// chunk_prefill.cu — chunked (WY/UT) prefill on tcgen05 tensor cores.
// (Not yet available: chunked_supports() reports false, so GDN_ALGO_AUTO uses
// the token scan and GDN_ALGO_CHUNKED is refused on the host.)
#include "params.h"

namespace gdn {

bool chunked_supports(int32_t, int32_t, int32_t, int32_t, int) { return false; }

size_t chunked_workspace_bytes(int32_t, int64_t, int32_t, int32_t, int32_t, int32_t) { return 0; }

cudaError_t launch_chunked(const PrefillArgs&, cudaStream_t) { return cudaErrorNotSupported; }

}  // namespace gdn
