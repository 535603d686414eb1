// fp32 linear-layer backward and forward on the tensor cores from tf32
// halves (MODE 2 of tc_mmbwd_kernel): the launch logic.
//
// The fp32 path needs fp32-accurate products (llm.c dev/cuda/matmul_backward.cu
// turns TF32 off in its main for exactly that reason). A value x is split into
//   hi = x with its 13 low mantissa bits cleared   (a tf32 value, exactly)
//   lo = x - hi                                     (exact in fp32, |lo| < 2^-10 |x|)
// and x*y is formed as hi_x*hi_y + hi_x*lo_y + lo_x*hi_y: the dropped lo_x*lo_y
// and the tf32 reading of lo leave a relative error near 2^-20 per product,
// below fp32 accumulation error over the long reductions.
//
// Every product is D += A . B^T with both operands K-major in shared memory:
//   dinp    (BT x C) += dout (BT x OC) . weight (OC x C)     A K-major, B MN-major
//   dweight (OC x C) += dout^T (OC x BT) . inp (BT x C)      A and B MN-major
//   out     (BT x OC) += inp (BT x C) . weight^T              A and B K-major
// The kernel loads the raw fp32 tensors by TMA and its split warps write the
// two planes of every stage (transposing the MN-major ones), so nothing is
// copied in global memory and the path needs no workspace. dbias (the column
// sums of dout) comes from the same split warps, which see every element of
// dout once on the dweight items of the first column tile.
#include "../../include/mmbwd.h"
#include "internal.h"
#include "ops.h"

namespace mmbwd {

bool x3_shape_ok(int64_t BT, int64_t C, int64_t OC) {
    // rows of 16-byte multiples for the tensor maps and the epilogue's 4-column vectors
    return BT > 0 && C > 0 && OC > 0 && C % 4 == 0 && OC % 4 == 0;
}

cudaError_t x3_launch(float* dinp, float* dweight, float* dbias, const float* dout, const float* inp,
                      const float* weight, int64_t BT, int64_t C, int64_t OC, int num_sms, cudaStream_t stream) {
    if (take_injected_launch_failure()) return cudaErrorLaunchFailure;
    // Both products in one launch where it fits (their tiles share the CTA
    // pairs, longest first, instead of each launch ending on a partial wave)
    static thread_local TcPlan pp;
    pp = tc_make_plan_x3_pair(BT, C, OC, num_sms);
    if (pp.n_items > 0) return tc_launch_x3_pair(pp, dinp, dweight, dbias, dout, inp, weight, BT, C, OC, stream);
    // dinp (BT x C) += dout . weight, K = OC
    const TcPlan p1 = tc_make_plan_x3(BT, C, OC, num_sms);
    cudaError_t e = tc_launch_x3(p1, dinp, dout, false, OC, weight, true, C, BT, C, OC, nullptr, stream);
    if (e != cudaSuccess) return e;
    // dweight (OC x C) += dout^T . inp, K = BT, and dbias
    const TcPlan p2 = tc_make_plan_x3(OC, C, BT, num_sms);
    return tc_launch_x3(p2, dweight, dout, true, OC, inp, true, C, OC, C, BT, dbias, stream);
}

// The forward out = inp . weight^T + bias on the same path: out is first set
// to the bias (or zero) and the product is then added to it.
bool x3_forward_shape_ok(int64_t BT, int64_t C, int64_t OC) {
    return BT > 0 && C > 0 && OC > 0 && OC % 4 == 0 && C % 4 == 0;
}

cudaError_t x3_forward_launch(float* out, const float* inp, const float* weight, const float* bias, int64_t BT,
                              int64_t C, int64_t OC, int num_sms, cudaStream_t stream) {
    if (take_injected_launch_failure()) return cudaErrorLaunchFailure;
    cudaError_t e = fill_rows_launch(out, bias, BT, OC, MMBWD_F32, stream);
    if (e != cudaSuccess) return e;
    const TcPlan p = tc_make_plan_x3(BT, OC, C, num_sms);
    return tc_launch_x3(p, out, inp, false, C, weight, false, C, BT, OC, C, nullptr, stream);
}

}  // namespace mmbwd
