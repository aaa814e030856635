// Scale-factor transform: FP32 scales -> MN-major, TMA-aligned layout.
//
// PaperTrace "02 · DeepGEMM 技术解析" §3.1-3.2 and "DeepSeek V4 源码剖析 第13章"
// §13.3: the packed form keeps the 8 exponent bits of each FP32 scale
// ((bits >> 23) & 0xff, so a non-power-of-two scale is truncated: 0.75 -> 0.5),
// puts four consecutive K-groups in one int32 little-endian by K, and stores the
// words MN-major with a K-slice stride of align(mn, 4) words; the scale rows are
// broadcast from gran_mn to one per MN index.  Memory bound: one thread per
// output word, consecutive threads write consecutive MN rows (coalesced).
// Launched as programmatic dependents: a kernel lets the next grid start its
// prologue at once and waits for the previous one before touching memory.
#include "dg_internal.h"
#include "ptx.cuh"

namespace dg {

__global__ void __launch_bounds__(256) dg_transform_sf_packed_kernel(
    const float *__restrict__ sf, int mn_rows, int sf_k, int gran_mn, int mn, int psf_k,
    int stride, uint32_t *__restrict__ out, int32_t *status) {
    grid_launch_dependents();
    grid_dependency_wait();
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    const int pslice = blockIdx.y;
    const int b = blockIdx.z;
    uint32_t word = 0;
    bool inexact = false;
    if (i < mn) {
        const float *row = sf + (static_cast<int64_t>(b) * mn_rows + i / gran_mn) * sf_k;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int k = 4 * pslice + j;
            if (k < sf_k) {
                const uint32_t bits = __float_as_uint(__ldg(row + k));
                word |= ((bits >> 23) & 0xFFu) << (8 * j);
                inexact |= (bits & 0x807FFFFFu) != 0u;
            }
        }
    }
    if (i < stride) out[(static_cast<int64_t>(b) * psf_k + pslice) * stride + i] = word;
    if (status != nullptr) {
        const unsigned any = __ballot_sync(0xFFFFFFFFu, inexact);
        if (any != 0u && (threadIdx.x & 31) == 0) atomicOr(status, DG_DEV_INEXACT_SCALE);
    }
}

__global__ void __launch_bounds__(256) dg_transform_sf_f32_kernel(
    const float *__restrict__ sf, int mn_rows, int sf_k, int gran_mn, int mn, int stride,
    float *__restrict__ out) {
    grid_launch_dependents();
    grid_dependency_wait();
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    const int k = blockIdx.y;
    const int b = blockIdx.z;
    if (i >= stride) return;
    float v = 0.0f;
    if (i < mn) v = __ldg(sf + (static_cast<int64_t>(b) * mn_rows + i / gran_mn) * sf_k + k);
    out[(static_cast<int64_t>(b) * sf_k + k) * stride + i] = v;
}

// K-grouped scales (PaperTrace "02 · DeepGEMM 技术解析" §3.3): the input is
// FP32 [rows][mn], one row per 128-K block of the concatenated groups, mn
// contiguous; each group's rows are packed on their own, 4 per word (byte j =
// the group's row 4q + j, 0 past its last row), and the groups' packed rows
// follow one another.  One thread per output word; consecutive threads take
// consecutive MN indices.
__global__ void __launch_bounds__(256) dg_transform_sf_k_grouped_kernel(
    const float *__restrict__ sf, int mn, const __grid_constant__ KGroupRows t, uint32_t *__restrict__ out,
    int32_t *status) {
    grid_launch_dependents();
    grid_dependency_wait();
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    const int prow = blockIdx.y;
    // the group holding packed row prow: prow[e] <= prow < prow[e + 1] (empty
    // groups have prow[e] == prow[e + 1] and are skipped)
    int lo = 0, hi = t.num_groups;   // number of e in [1, num_groups] with t.prow[e] <= prow
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (t.prow[mid] <= prow) lo = mid; else hi = mid - 1;
    }
    const int e = lo;
    const int r0 = t.srow[e] + 4 * (prow - t.prow[e]);
    const int nrow = t.srow[e + 1] - r0;
    uint32_t word = 0;
    bool inexact = false;
    if (i < mn) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            if (j < nrow) {
                const uint32_t bits = __float_as_uint(__ldg(sf + static_cast<int64_t>(r0 + j) * mn + i));
                word |= ((bits >> 23) & 0xFFu) << (8 * j);
                inexact |= (bits & 0x807FFFFFu) != 0u;
            }
        }
        out[static_cast<int64_t>(prow) * mn + i] = word;
    }
    if (status != nullptr) {
        const unsigned any = __ballot_sync(0xFFFFFFFFu, inexact);
        if (any != 0u && (threadIdx.x & 31) == 0) atomicOr(status, DG_DEV_INEXACT_SCALE);
    }
}

cudaError_t launch_transform_sf_k_grouped(const float *sf, int mn, const KGroupRows &t, int packed_rows,
                                          void *out, int32_t *status, cudaStream_t stream) {
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.blockDim = dim3(256);
    cfg.gridDim = dim3((mn + 255) / 256, packed_rows, 1);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, dg_transform_sf_k_grouped_kernel, sf, mn, t, static_cast<uint32_t *>(out),
                              status);
}

cudaError_t launch_transform_sf(const float *sf, int batch, int mn_rows, int sf_k, int gran_mn,
                                int mn, int out_fmt, void *out, int32_t *status,
                                cudaStream_t stream) {
    const int stride = (mn + 3) / 4 * 4;
    const int psf_k = (sf_k + 3) / 4;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.blockDim = dim3(256);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (out_fmt == DG_SF_UE8M0_PACKED) {
        cfg.gridDim = dim3((stride + 255) / 256, psf_k, batch);
        return cudaLaunchKernelEx(&cfg, dg_transform_sf_packed_kernel, sf, mn_rows, sf_k, gran_mn, mn, psf_k,
                                  stride, static_cast<uint32_t *>(out), status);
    }
    cfg.gridDim = dim3((stride + 255) / 256, sf_k, batch);
    return cudaLaunchKernelEx(&cfg, dg_transform_sf_f32_kernel, sf, mn_rows, sf_k, gran_mn, mn, stride,
                              static_cast<float *>(out));
}

}  // namespace dg
