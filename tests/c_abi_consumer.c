/* A plain C99 consumer of libmoeprefill.so: it includes only
 * include/moe_prefill.h (no C++, CUDA or torch headers), links the library,
 * and calls the entry points that need no GPU -- sizes, host-side argument
 * validation and status text -- printing what they return. */
#include <stdio.h>
#include <string.h>

#include "moe_prefill.h"

int main(void) {
  MoeLayerDesc d;
  MoeLayerDesc bad;
  size_t ws, io, ws_bad;
  int64_t tiled;
  int rc_null, rc_shape;

  memset(&d, 0, sizeof d);
  d.T = 16384;
  d.d = 2560;
  d.n_ff = 640;
  d.E = 512;
  d.k = 10;
  d.gu_fmt = MOE_FMT_W2;
  d.down_fmt = MOE_FMT_W4NL;
  d.gu_layout = MOE_GU_INTERLEAVED;
  ws = moe_prefill_workspace_bytes(&d);
  tiled = moe_tiled_pack_bytes(&d);
  io = moe_host_io_bytes(&d);

  bad = d;
  bad.d = 100; /* not a multiple of 128 */
  ws_bad = moe_prefill_workspace_bytes(&bad);

  rc_null = moe_prefill_layer(NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL, 0, NULL);
  rc_shape = moe_route(&bad, NULL, NULL, 0, NULL);

  printf("%zu %lld %zu %zu %d %d %s\n", ws, (long long)tiled, io, ws_bad, rc_null, rc_shape,
         moe_status_string(MOE_ERR_SHAPE));
  return 0;
}
