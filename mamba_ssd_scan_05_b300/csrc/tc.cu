// tc.cu -- tensor-core (tcgen05) path: not built yet in this revision.
#include "common.cuh"

namespace ssd {
bool tc_supports(int32_t, int64_t, int64_t, int) { return false; }
size_t tc_workspace_bytes(int64_t, int64_t, int64_t, int64_t, int64_t, int) {
    return kWsHeaderBytes;
}
int tc_launch(const ScanArgs&) { return SSD_ERR_UNSUPPORTED; }
}  // namespace ssd
