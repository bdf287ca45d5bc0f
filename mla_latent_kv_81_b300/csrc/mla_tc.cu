// Tensor-core projection paths not specialised yet: those calls take the SIMT path.
#include "mla_tc.cuh"

namespace mla {

bool tc_compress_supported(const mla_config*, int) { return false; }
size_t tc_compress_workspace_bytes(const mla_config*, int) { return 0; }
cudaError_t tc_compress_append(const Ctx&, const mla_config*, const void*, const void*, const void*, const int32_t*,
                               const int32_t*, const mla_rope_table&, const mla_paged_cache&, int, void*) {
  return cudaErrorNotSupported;
}
bool tc_absorb_supported(const mla_config*, int) { return false; }
size_t tc_absorb_workspace_bytes(const mla_config*, int) { return 0; }
cudaError_t tc_absorb_query(const Ctx&, const mla_config*, const void*, const void*, const void*, const void*,
                            const int32_t*, const mla_rope_table&, void*, int, void*) { return cudaErrorNotSupported; }
bool tc_output_supported(const mla_config*, int) { return false; }
size_t tc_output_workspace_bytes(const mla_config*, int) { return 0; }
cudaError_t tc_output_project(const Ctx&, const mla_config*, const void*, const void*, const void*, void*, int,
                              void*) { return cudaErrorNotSupported; }

}  // namespace mla
