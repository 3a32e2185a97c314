// Host orchestration of the tcgen05 tensor-core path (placeholder until the
// kernels land).
#include "fs_host.cuh"

namespace fs {

int64_t workspace_bytes_tc(int64_t, int64_t, int32_t, int32_t, int, const fs_options*) { return -1; }

fs_status solve_tc(Call&, Problem&, int32_t, const fs_options*) {
    return fail(FS_ERR_UNSUPPORTED, "tensor-core path not built");
}

fs_status apply_tc(Call&, Problem&, int, const fs_options*) {
    return fail(FS_ERR_UNSUPPORTED, "tensor-core path not built");
}

}  // namespace fs
