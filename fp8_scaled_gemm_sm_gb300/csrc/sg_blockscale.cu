// sg_blockscale.cu -- placeholder until the promotion kernel lands.
#include "sg_internal.h"
namespace sg {
cudaError_t blockscale_prepare() { return cudaSuccess; }
sg_status_t blockscale_launch(const LaunchArgs&) { return SG_ERR_UNSUPPORTED_SHAPE; }
void blockscale_config(TileConfig* c) { c->bm = 128; c->bn = 128; c->bk = 128; c->stages = 4; }
}  // namespace sg
