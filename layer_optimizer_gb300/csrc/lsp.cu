// Placeholder: the sparse-projector kernels land in the next change.
#include "common.h"

struct lsp_projector_s { int64_t rows; int32_t d, k; };

extern "C" {
sf_status lsp_projector_create(int64_t, int32_t, int32_t, const int32_t*, const float*, int, void*,
                               lsp_projector* out) {
  if (out) *out = nullptr;
  return sf::fail(SF_ERR_UNSUPPORTED, "not built yet");
}
sf_status lsp_projector_export_csc(lsp_projector, int32_t*, int32_t*, float*, int32_t*, void*) {
  return sf::fail(SF_ERR_UNSUPPORTED, "not built yet");
}
int64_t lsp_projector_rows(lsp_projector p) { return p ? p->rows : -1; }
int32_t lsp_projector_dim(lsp_projector p) { return p ? p->d : -1; }
int32_t lsp_projector_nnz_per_row(lsp_projector p) { return p ? p->k : -1; }
sf_status lsp_projector_destroy(lsp_projector p) { delete p; return SF_OK; }
size_t lsp_workspace_bytes(int64_t, int64_t, int32_t) { return 0; }
sf_status lsp_compress(lsp_projector, lsp_projector, const void*, sf_dtype, int64_t, int64_t, float*,
                       void*, size_t, void*) {
  return sf::fail(SF_ERR_UNSUPPORTED, "not built yet");
}
sf_status lsp_decompress_apply(lsp_projector, lsp_projector, const float*, void*, sf_dtype, void*,
                               int64_t, int64_t, void*, size_t, void*) {
  return sf::fail(SF_ERR_UNSUPPORTED, "not built yet");
}
}
