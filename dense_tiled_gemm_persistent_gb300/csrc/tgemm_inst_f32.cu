// Compiled variants of the persistent GEMM kernel with F32 output.
// Each entry: output tile width BN, ring depth STAGES, output type, B layout
// (0 = B stored N x K, K-major; 1 = B stored K x N, MN-major); the pair
// entries run 256 x 256 tiles on CTA pairs; the skinny entries are the
// swap-AB split-K kernels for at most 64 rows of A (global-workspace and
// in-cluster reductions) and the in-cluster one for 65-128 rows, by padded
// row count; the quad entries run two pairs
// that share A (clusters of four); the last eight take FP8 and FP32-as-TF32
// operands (B stored N x K).
#include "tgemm_kernel_quad.cuh"
#include "tgemm_kernel_skinny.cuh"
#include "tgemm_kernel_splitk_cluster.cuh"

namespace tgemm {

const KernelVariant kVariantsF32[] = {
    TGEMM_VARIANT(256, 4, OUT_F32, 0),
    TGEMM_VARIANT(256, 4, OUT_F32, 1),
    TGEMM_VARIANT(128, 6, OUT_F32, 0),
    TGEMM_VARIANT(128, 6, OUT_F32, 1),
    TGEMM_VARIANT(128, 2, OUT_F32, 0),
    TGEMM_VARIANT(128, 2, OUT_F32, 1),
    TGEMM_PAIR_VARIANT(6, OUT_F32, 0),
    TGEMM_PAIR_VARIANT(6, OUT_F32, 1),
    TGEMM_SKINNY_VARIANT(16, OUT_F32, 0),
    TGEMM_SKINNY_VARIANT(16, OUT_F32, 1),
    TGEMM_SKINNY_VARIANT(32, OUT_F32, 0),
    TGEMM_SKINNY_VARIANT(32, OUT_F32, 1),
    TGEMM_SKINNY_VARIANT(64, OUT_F32, 0),
    TGEMM_SKINNY_VARIANT(64, OUT_F32, 1),
    TGEMM_CLUSTER_SPLIT_VARIANT(16, OUT_F32, 0),
    TGEMM_CLUSTER_SPLIT_VARIANT(16, OUT_F32, 1),
    TGEMM_CLUSTER_SPLIT_VARIANT(32, OUT_F32, 0),
    TGEMM_CLUSTER_SPLIT_VARIANT(32, OUT_F32, 1),
    TGEMM_CLUSTER_SPLIT_VARIANT(64, OUT_F32, 0),
    TGEMM_CLUSTER_SPLIT_VARIANT(64, OUT_F32, 1),
    TGEMM_CLUSTER_SPLIT_VARIANT_RING(128, OUT_F32, 0, 216),
    TGEMM_CLUSTER_SPLIT_VARIANT_RING(128, OUT_F32, 1, 216),
    TGEMM_QUAD_VARIANT(6, OUT_F32, 0),
    TGEMM_QUAD_VARIANT(6, OUT_F32, 1),
    TGEMM_VARIANT_KIND(256, 4, OUT_F32, KIND_F8),
    TGEMM_VARIANT_KIND(128, 6, OUT_F32, KIND_F8),
    TGEMM_PAIR_VARIANT_KIND(6, OUT_F32, KIND_F8),
    TGEMM_QUAD_VARIANT_KIND(6, OUT_F32, KIND_F8),
    TGEMM_CLUSTER_SPLIT_VARIANTS_F8(OUT_F32),
    TGEMM_VARIANT_KIND(256, 4, OUT_F32, KIND_TF32),
    TGEMM_VARIANT_KIND(128, 6, OUT_F32, KIND_TF32),
    TGEMM_PAIR_VARIANT_KIND(6, OUT_F32, KIND_TF32),
    TGEMM_QUAD_VARIANT_KIND(6, OUT_F32, KIND_TF32),
};
const int kNumVariantsF32 = (int)(sizeof(kVariantsF32) / sizeof(kVariantsF32[0]));

}  // namespace tgemm
