// Streaming path of libspecverify (persistent grid). Not yet built: the
// library routes every call to the rowwise path until it is.
#include "sv_internal.h"

namespace sv {

bool streaming_applicable(const Args&) { return false; }
size_t streaming_workspace_bytes(int, int, int, int, int) { return 256; }
int streaming_default_grid(const DeviceInfo& dev) { return dev.num_sms; }
cudaError_t launch_streaming(const Args&, const DeviceInfo&, int, void*, size_t, cudaStream_t) {
    return cudaErrorNotSupported;
}

}  // namespace sv
