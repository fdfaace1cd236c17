// Host-side window-assignment arithmetic (TERRA Sec. V.A): the padding that
// the fixed round-robin assignment needs, Eq. (3). No device code.
#include <cstdint>

#include "swin_attn.h"

int swin_attn_fixed_padded_extent(int64_t extent, int64_t stride, int64_t window, int64_t ranks,
                                  int64_t *padded) {
  if (!padded || extent < 1 || stride < 1 || window < 1 || ranks < 1) return SWIN_ERR_INVALID_ARG;
  if (stride > INT64_MAX / window) return SWIN_ERR_INVALID_ARG;
  int64_t q = stride * window;  // input points per window
  if (q > INT64_MAX / ranks) return SWIN_ERR_INVALID_ARG;
  q *= ranks;  // input points per row of windows across the mesh dimension
  const int64_t blocks = extent / q + (extent % q != 0);
  if (blocks > INT64_MAX / q) return SWIN_ERR_INVALID_ARG;
  *padded = blocks * q;
  return SWIN_OK;
}
