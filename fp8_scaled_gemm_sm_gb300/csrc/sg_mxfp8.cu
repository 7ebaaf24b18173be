// sg_mxfp8.cu -- placeholder until the block-scaled kernel lands.
#include "sg_internal.h"
namespace sg {
cudaError_t mxfp8_prepare() { return cudaSuccess; }
sg_status_t mxfp8_launch(const LaunchArgs&) { return SG_ERR_UNSUPPORTED_SHAPE; }
void mxfp8_config(TileConfig* c) { c->bm = 128; c->bn = 224; c->bk = 128; c->stages = 4; }
}  // namespace sg
