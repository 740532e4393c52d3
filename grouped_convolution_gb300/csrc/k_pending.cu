// k_pending.cu -- schedules not yet specialised: never selected.
#include "gconv_internal.h"

namespace gconv {
namespace {
bool no(const gconv_desc &, const Ptrs &) { return false; }
cudaError_t none(const Params &, const Ptrs &, cudaStream_t, int *) { return cudaErrorNotSupported; }
}  // namespace
const Schedule kDwMult = {"dw_mult", no, none};
const Schedule kGrpPlane = {"grp_plane", no, none};
const Schedule kGrpReduce = {"grp_reduce", no, none};
}  // namespace gconv
