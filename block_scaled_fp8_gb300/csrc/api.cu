// Host side of the C ABI: argument validation, TMA descriptors, tile-shape
// choice and kernel launch.  Declarations and contracts are in include/dg.h.
#include <atomic>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "dg_internal.h"

namespace dg {
namespace {

// ------------------------------------------------------------------ settings

std::atomic<int> g_num_sms_override{0};
std::atomic<int> g_timeout_ms{2000};
std::atomic<uint32_t> g_debug_flags{0};
thread_local int g_last_config[6] = {0, 0, 0, 0, 0, 0};

constexpr int kMaxDevices = 64;
struct DeviceInfo {
    int checked = 0;     // 0 unknown, 1 ok, -1 unsupported
    int num_sms = 0;
};
DeviceInfo g_devices[kMaxDevices];
std::mutex g_dev_mutex;

// cuTensorMapEncodeTiled, reached through the runtime so that the library does
// not link libcuda directly.
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;
std::once_flag g_encode_once;

EncodeTiledFn get_encode() {
    std::call_once(g_encode_once, [] {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<EncodeTiledFn>(fn);
    });
    return g_encode;
}

// Current device must be an sm_103 GPU; fills its SM count.
dg_status check_device(int *num_sms) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return DG_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_dev_mutex);
    DeviceInfo &di = g_devices[dev];
    if (di.checked == 0) {
        int major = 0, minor = 0, sms = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return DG_ERR_CUDA;
        di.checked = (major == 10 && minor == 3) ? 1 : -1;
        di.num_sms = sms;
    }
    if (di.checked < 0) return DG_ERR_UNSUPPORTED;
    int ov = g_num_sms_override.load();
    *num_sms = (ov > 0 && ov < di.num_sms) ? ov : di.num_sms;
    return DG_OK;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
int64_t cdiv64(int64_t a, int64_t b) { return (a + b - 1) / b; }
int64_t align4(int64_t x) { return (x + 3) / 4 * 4; }

bool encode_2d(CUtensorMap *map, CUtensorMapDataType dtype, int elem_bytes, const void *base,
               uint64_t dim0, uint64_t dim1, uint64_t stride1_bytes, uint32_t box0, uint32_t box1,
               CUtensorMapSwizzle swizzle, CUtensorMapL2promotion promo) {
    EncodeTiledFn enc = get_encode();
    if (enc == nullptr) return false;
    (void)elem_bytes;
    cuuint64_t dims[2] = {dim0, dim1};
    cuuint64_t strides[1] = {stride1_bytes};
    cuuint32_t box[2] = {box0, box1};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(map, dtype, 2, const_cast<void *>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, promo,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// K-blocked 3-D view of a K-contiguous FP8 operand [rows][ld]: x = K within a
// 128-K block, y = row, z = K-block (stride 128 bytes).  A box {128, box_rows,
// depth} loads `depth` consecutive K-blocks as consecutive 128B-swizzled
// [box_rows][128] slabs, i.e. the stages of one ring slot.  Valid only when K
// is a multiple of 128 (x never runs past K inside a block).
bool encode_kblocked_3d(CUtensorMap *map, const void *base, uint64_t rows, uint64_t ld_bytes,
                        uint64_t k_blocks, uint32_t box_rows, uint32_t depth) {
    EncodeTiledFn enc = get_encode();
    if (enc == nullptr) return false;
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(kBlockK), rows, k_blocks};
    cuuint64_t strides[2] = {ld_bytes, static_cast<cuuint64_t>(kBlockK)};
    cuuint32_t box[3] = {static_cast<cuuint32_t>(kBlockK), box_rows, depth};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void *>(base), dims, strides,
                     box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// Block-N values compiled into the block-scaled kernel family.
constexpr int kBsBlockN[] = {16, 32, 48, 64, 96, 128, 160, 176, 192, 224, 256};
constexpr int kMaxBlockNWithC = 160;

// Tile-shape choice: maximise the fraction of SM-time spent on useful tiles
// (wave quantisation x N padding) weighted by a per-tile efficiency that grows
// with BLOCK_N (larger tiles re-read less operand data per FLOP).  Split-K is
// never used: with few M blocks, narrow BLOCK_N is what fills the SMs (the
// non-power-of-two block idea of "02 · DeepGEMM 技术解析" §4.3).
int choose_block_n(int64_t m_blocks, int n, int num_sms, bool with_c, bool count_waves) {
    static const int forced_bn = [] {
        const char *e = std::getenv("DG_BLOCK_N");
        return e ? std::atoi(e) : 0;
    }();
    double best = -1.0;
    int best_bn = 128;
    for (int bn : kBsBlockN) {
        if (with_c && bn > kMaxBlockNWithC) continue;
        if (forced_bn && bn != forced_bn) continue;
        const int64_t nb = cdiv64(n, bn);
        const int64_t tiles = m_blocks * nb;
        const int64_t waves = cdiv64(tiles, num_sms);
        // (masked layouts: the row blocks come from masked_m on the device, so the tile
        // count and its waves are unknown here; the weight stream sets the time)
        const double wave_eff = count_waves ? static_cast<double>(tiles) / static_cast<double>(waves * num_sms) : 1.0;
        const double pad_eff = static_cast<double>(n) / static_cast<double>(nb * bn);
        const double tile_eff = static_cast<double>(bn) / (bn + 64.0);
        const double score = wave_eff * pad_eff * tile_eff;
        if (score > best + 1e-9) {
            best = score;
            best_bn = bn;
        }
    }
    return best_bn;
}

__global__ void dg_fill_d_kernel(const uint16_t *c, int64_t ldc, uint16_t *d, int64_t ldd, int m,
                                 int n) {
    const int64_t total = static_cast<int64_t>(m) * n;
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t r = i / n, col = i % n;
        d[r * ldd + col] = c ? c[r * ldc + col] : static_cast<uint16_t>(0);
    }
}

__global__ void dg_fill_d_f32_kernel(const float *c, int64_t ldc, float *d, int64_t ldd, int m, int n) {
    const int64_t total = static_cast<int64_t>(m) * n;
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t r = i / n, col = i % n;
        d[r * ldd + col] = c ? c[r * ldc + col] : 0.0f;
    }
}

// Operand views of one block-scaled launch (all 2-D, K or MN contiguous).
struct BsOperands {
    const void *a;  int64_t lda;  uint64_t a_rows;
    const void *b;  int64_t ldb;  uint64_t b_rows;
    const void *sfa; uint64_t sfa_mn; uint64_t sfa_slices;  // inner = MN rows, outer = K slices
    const void *sfb; uint64_t sfb_mn; uint64_t sfb_slices;
    void *d;        int64_t ldd;  uint64_t d_rows;
};

// 256-row CTA pairs (cta_group::2) unless DG_DEBUG_SINGLE_CTA is set: dense
// problems with more than one 128-row block; contiguous layouts of at most
// kMaxPairPrefix m-pairs (and fewer than 2^15 experts); masked layouts of at
// most kMaxPairPrefix experts that expect more than 256 rows per expert.  The
// masked decode (a few dozen rows per expert) is bound by reading each
// expert's B once from HBM, which the single-CTA kernel does as well (its two
// 128-row blocks of an expert share B through L2) at less cost per tile.
bool use_pair_kernel(const GemmParams &p, int64_t m_blocks_hint) {
    if (g_debug_flags.load() & DG_DEBUG_SINGLE_CTA) return false;
    if (p.mode == kModeDense) return p.rows > kBlockM;
    if (p.mode == kModeContiguous)
        return cdiv64(p.rows, 2 * kBlockM) <= kMaxPairPrefix && p.num_groups < 32768;
    return p.rows > kBlockM && p.num_groups <= kMaxPairPrefix && m_blocks_hint > 2LL * p.num_groups;
}

int cached_max_pairs(int bn, bool with_c, int mp, bool f32 = false, int lay = 0) {
    static std::mutex mu;
    static int cache[kMaxDevices][2][2][2][16][513];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices || bn <= 0 || bn > 512) return 0;
    std::lock_guard<std::mutex> lock(mu);
    int &v = cache[dev][with_c ? 1 : 0][mp == 128 ? 1 : 0][f32 ? 1 : 0][lay & 15][bn];
    if (v == 0) v = bs2_max_active_pairs(bn, with_c, mp, f32, lay & 15);
    return v;
}

int usable_pairs(int bn, bool with_c, int mp, int num_sms, bool f32 = false, int lay = 0) {
    int pairs = cached_max_pairs(bn, with_c, mp, f32, lay);
    if (pairs * 2 > num_sms) pairs = num_sms / 2;
    return pairs;
}

// BLOCK_N of the 256-row pair kernel: the score of choose_block_n over the
// co-resident pairs (DG_PAIR_BLOCK_N forces one); m_pairs is the expected
// number of 256-row units.
int choose_pair_block_n(const GemmParams &p, bool with_c, int64_t m_pairs, int num_sms) {
    int bn = 0;
    double best = -1.0;
    static const int forced_bn = [] {
        const char *e = std::getenv("DG_PAIR_BLOCK_N");
        return e ? std::atoi(e) : 0;
    }();
    const bool f32 = p.d_f32 != nullptr;
    if ((g_debug_flags.load() & DG_DEBUG_WIDE_PAIR) && !with_c && !f32) {
        KernelInfo ki;
        if (get_bs2_kernel_info(384, false, 256, &ki) && usable_pairs(384, false, 256, num_sms) > 0) return 384;
    }
    for (int cand : {128, 192, 224, 240, 256, 384}) {
        if (forced_bn && cand != forced_bn) continue;
        // 384-column tiles: dense GEMMs only (3 % slower on the contiguous MoE shape
        // with N=4096, K=7168)
        if (cand > 256 && p.mode != kModeDense && !forced_bn) continue;
        KernelInfo ki;
        if (!get_bs2_kernel_info(cand, with_c, 256, &ki, f32)) continue;
        const int pairs = usable_pairs(cand, with_c, 256, num_sms, f32);
        if (pairs <= 0) continue;
        const int64_t nb = cdiv64(p.n, cand);
        const int64_t tiles = m_pairs * nb;
        const int64_t waves = cdiv64(tiles, pairs);
        double score = static_cast<double>(tiles) / static_cast<double>(waves * pairs) *
                       static_cast<double>(p.n) / static_cast<double>(nb * cand) * (cand / (cand + 64.0));
        // with one accumulator the MMAs stop for about 1.5 K-blocks per tile while the
        // epilogue reads the accumulator out
        if (ki.num_acc == 1) score *= 1.0 - 1.5 / static_cast<double>(cdiv64(p.k, kBlockK));
        if (score > best + 1e-9) { best = score; bn = cand; }
    }
    return bn;
}

// Skinny dense problems (one 128-row block, no C): the single-CTA kernel with
// BLOCK_N bn1, or the 128-row pair kernel, whose CTAs load 64 rows of A each.
// With one row block every CTA re-reads the same A tile, and a CTA's loads are
// capped near 60 bytes per cycle (a load-only probe; ~48 with the MMAs reading
// shared memory beside them), so the time of a K-block is modelled as
// max(bytes a CTA loads / 60, MMA cycles) times the waves of tiles.  Returns
// the pair kernel's BLOCK_N, or 0 to keep the single-CTA kernel.
int choose_skinny_pair_block_n(const GemmParams &p, int bn1, int num_sms) {
    static const int forced = [] {
        const char *e = std::getenv("DG_SKINNY_PAIR_BLOCK_N");
        return e ? std::atoi(e) : 0;
    }();
    if (forced < 0) return 0;
    if (forced > 0) return usable_pairs(forced, false, 128, num_sms) > 0 ? forced : 0;
    auto cost = [](int64_t waves, double bytes, double mma) {
        return static_cast<double>(waves) * (bytes / 60.0 > mma ? bytes / 60.0 : mma);
    };
    const double mma1 = 2.0 * bn1 > 200.0 ? 2.0 * bn1 : 200.0;
    const double cost1 = cost(cdiv64(cdiv64(p.n, bn1), num_sms), kBlockM * kBlockK + bn1 * kBlockK, mma1);
    int best_bn = 0;
    double best = cost1 * 0.95;   // switch only for a clear gain
    for (int cand : {32, 64, 96, 128}) {
        const int pairs = usable_pairs(cand, false, 128, num_sms);
        if (pairs <= 0) continue;
        const double mma2 = cand > 200 ? cand : 200.0;
        const double c = cost(cdiv64(cdiv64(p.n, cand), pairs), kBlockM / 2 * kBlockK + cand / 2 * kBlockK, mma2);
        if (c < best) { best = c; best_bn = cand; }
    }
    return best_bn;
}

// The packed scale words are read by the kernels' scale warps (cp.async), not by TMA.
void set_scale_words(GemmParams &p, const BsOperands &o) {
    p.sfa_words = static_cast<const uint32_t *>(o.sfa);
    p.sfb_words = static_cast<const uint32_t *>(o.sfb);
    p.sfa_ld = static_cast<int>(align4(o.sfa_mn));
    p.sfb_ld = static_cast<int>(align4(o.sfb_mn));
    p.sfa_slices = static_cast<int>(o.sfa_slices);
    p.sfb_slices = static_cast<int>(o.sfb_slices);
}

// One launch of the pair kernel with mp rows per pair tile and BLOCK_N bn;
// max_units bounds the number of mp-row units (the grid size).
dg_status launch_pair(GemmParams &p, const BsOperands &o, int mp, int bn, int64_t max_units,
                      int num_sms, cudaStream_t stream) {
    // FP32 D: the caller sets d_f32 (and c_f32 for an FP32 C) before the call
    const bool f32 = p.d_f32 != nullptr;
    const bool with_c = f32 ? p.c_f32 != nullptr : p.c != nullptr;
    const int lay = p.layout;   // bit 0 A MN-major, bit 1 B MN-major, bit 2 B FP4
    KernelInfo info;
    if (bn == 0 || !get_bs2_kernel_info(bn, with_c, mp, &info, f32, lay)) return DG_ERR_UNSUPPORTED;
    const int pairs = usable_pairs(bn, with_c, mp, num_sms, f32, lay);
    if (pairs <= 0) return DG_ERR_UNSUPPORTED;
    const uint32_t a_rows = static_cast<uint32_t>(mp / 2);   // rows of A each CTA loads
    TensorMaps maps;
    const int k = p.k;
    bool ok = true;
    // K a multiple of 128: one 3-D load per operand fills a ring slot
    p.ab_3d = (lay == 0 && k % kBlockK == 0 && info.group_kb > 1) ? 1 : 0;
    // a tile wider than 256 columns runs two MMAs (256 and bn - 256 columns); each CTA
    // loads half of each one's B rows through its own map
    const uint32_t b1_rows = static_cast<uint32_t>((bn > 256 ? 256 : bn) / 2);
    const uint32_t b2_rows = static_cast<uint32_t>(bn > 256 ? (bn - 256) / 2 : 0);
    if (p.ab_3d) {
        const uint64_t kblocks = static_cast<uint64_t>(k / kBlockK);
        ok &= encode_kblocked_3d(&maps.a, o.a, o.a_rows, o.lda, kblocks, a_rows, info.group_kb);
        ok &= encode_kblocked_3d(&maps.b, o.b, o.b_rows, o.ldb, kblocks, b1_rows, info.group_kb);
        if (b2_rows) ok &= encode_kblocked_3d(&maps.b2, o.b, o.b_rows, o.ldb, kblocks, b2_rows, info.group_kb);
    } else {
        // an MN-major operand ([K][MN], MN contiguous): boxes of 128 MN-bytes x G K-blocks of rows
        const uint32_t k_rows = static_cast<uint32_t>(info.group_kb * kBlockK);
        if (lay & 1)
            ok &= encode_2d(&maps.a, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, o.a, o.a_rows, k, o.lda, a_rows, k_rows,
                            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B);
        else
            ok &= encode_2d(&maps.a, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, o.a, k, o.a_rows, o.lda, kBlockK,
                            a_rows, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B);
        if (lay & 4)   // FP4 B, K-contiguous, two codes per byte: boxes of 128 codes x rows
            ok &= encode_2d(&maps.b, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, 1, o.b, k, o.b_rows, o.ldb, kBlockK,
                            b1_rows, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B);
        else if (lay & 2)   // a whole 128-byte atom per CTA, of which the MMA reads bn/2 columns
            ok &= encode_2d(&maps.b, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, o.b, o.b_rows, k, o.ldb, 128, k_rows,
                            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B);
        else
            ok &= encode_2d(&maps.b, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, o.b, k, o.b_rows, o.ldb, kBlockK,
                            b1_rows, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B);
        if (b2_rows)
            ok &= encode_2d(&maps.b2, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, o.b, k, o.b_rows, o.ldb, kBlockK,
                            b2_rows, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B);
    }
    if (!b2_rows) maps.b2 = maps.b;   // not read
    // D store boxes: 32 rows of 32 bytes (16 bf16 columns), or 64 bytes (16 FP32 columns, or
    // 32 bf16 columns with C)
    if (f32)
        ok &= encode_2d(&maps.d, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, o.d, p.n, o.d_rows, o.ldd * 4, 16, 32,
                        CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_NONE);
    else if (with_c)   // the bf16 C epilogue stores two adjacent chunks per box
        ok &= encode_2d(&maps.d, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, o.d, p.n, o.d_rows, o.ldd * 2, 32,
                        32, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_NONE);
    else
        ok &= encode_2d(&maps.d, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, o.d, p.n, o.d_rows, o.ldd * 2, 16,
                        32, CU_TENSOR_MAP_SWIZZLE_32B, CU_TENSOR_MAP_L2_PROMOTION_NONE);
    // bf16 C of a dense GEMM whose tile is whole 32-column boxes: the kernel keeps the
    // C tile in shared memory, loaded by TMA (boxes of 32 rows x 32 columns, as D's)
    const bool c_tile = !f32 && with_c && mp == 256 && bn % 32 == 0 && bn <= 256;
    if (c_tile && p.mode != kModeDense) return DG_ERR_UNSUPPORTED;   // (that layout has no grouped prefix)
    p.c_tma = (c_tile && (reinterpret_cast<uintptr_t>(p.c) & 15u) == 0 && (p.ldc * 2) % 16 == 0) ? 1 : 0;
    if (p.c_tma)
        ok &= encode_2d(&maps.c, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, p.c, p.n, o.d_rows, p.ldc * 2, 32, 32,
                        CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B);
    else
        maps.c = maps.d;   // not read
    if (!ok) return DG_ERR_CUDA;
    set_scale_words(p, o);
    p.c_v8 = (p.c != nullptr && (reinterpret_cast<uintptr_t>(p.c) & 31u) == 0 && p.ldc % 16 == 0) ? 1 : 0;
    // dense and contiguous: the pair kernel counts mp-row m-units (masked: unused;
    // K-grouped: the caller sets the m-units of one group)
    if (p.mode == kModeDense || p.mode == kModeContiguous) p.num_m_blocks = static_cast<int>(cdiv64(p.rows, mp));
    p.num_n_blocks = static_cast<int>(cdiv64(p.n, bn));
    p.num_k_blocks = static_cast<int>(cdiv64(k, kBlockK));
    p.group_m = 8;
    if (f32) p.d_f32 = static_cast<float *>(o.d);
    else p.d = static_cast<uint16_t *>(o.d);
    p.ldd = o.ldd;
    p.c_in_place = (f32 && p.c_f32 != nullptr && p.c_f32 == p.d_f32 && p.ldc == p.ldd) ? 1 : 0;
    p.timeout_ns = static_cast<uint64_t>(g_timeout_ms.load()) * 1000000ull;
    uint32_t dbg = g_debug_flags.load();
    if (dbg & DG_DEBUG_DROP_ONE_LOAD) g_debug_flags.fetch_and(~static_cast<uint32_t>(DG_DEBUG_DROP_ONE_LOAD));
    p.debug_flags = dbg;
    const int64_t tiles = max_units * p.num_n_blocks;
    const int64_t used = tiles < pairs ? tiles : pairs;
    const int grid = static_cast<int>(2 * used);
    if ((dbg & DG_DEBUG_PRINT_CONFIGS) || std::getenv("DG_PRINT_CONFIGS"))
        std::fprintf(stderr, "[dg] pair rows=%d n=%d k=%d -> BLOCK_M=%d BLOCK_N=%d stages=%d smem=%d grid=%d\n",
                     p.rows, p.n, k, mp, bn, info.stages, info.smem_bytes, grid);
    g_last_config[0] = mp;
    g_last_config[1] = bn;
    g_last_config[2] = info.stages;
    g_last_config[3] = grid;
    g_last_config[4] = 2;
    g_last_config[5] = 1;
    cudaError_t e = launch_bs2_gemm(bn, mp, maps, p, grid, stream);
    return e == cudaSuccess ? DG_OK : DG_ERR_CUDA;
}

dg_status launch_block_scaled(GemmParams &p, const BsOperands &o, int64_t m_blocks_hint,
                              int64_t max_tiles_per_n_block, int num_sms, cudaStream_t stream) {
    if (use_pair_kernel(p, m_blocks_hint)) {
        // dense: 256-row m-pairs; grouped: about half the 128-row blocks (at most all of them)
        const int64_t units_hint = p.mode == kModeDense ? cdiv64(p.rows, 2 * kBlockM) : cdiv64(m_blocks_hint, 2);
        const int64_t max_units = p.mode == kModeDense ? units_hint : max_tiles_per_n_block;
        return launch_pair(p, o, 256, choose_pair_block_n(p, p.c != nullptr, units_hint, num_sms), max_units,
                           num_sms, stream);
    }
    const bool with_c = p.c != nullptr;
    const int bn = choose_block_n(m_blocks_hint, p.n, num_sms, with_c, p.mode != kModeMasked);
    if (p.mode == kModeDense && !with_c && p.rows <= kBlockM &&
        !(g_debug_flags.load() & DG_DEBUG_SINGLE_CTA)) {
        const int bn2 = choose_skinny_pair_block_n(p, bn, num_sms);
        if (bn2 > 0) return launch_pair(p, o, 128, bn2, cdiv64(p.rows, 128), num_sms, stream);
    }
    KernelInfo info;
    if (!get_bs_kernel_info(bn, with_c, &info)) return DG_ERR_UNSUPPORTED;
    TensorMaps maps;
    const int k = p.k;
    bool ok = true;
    // K a multiple of 128: one 3-D load per operand fills a ring slot
    p.ab_3d = (k % kBlockK == 0 && info.group_kb > 1) ? 1 : 0;
    if (p.ab_3d) {
        const uint64_t kblocks = static_cast<uint64_t>(k / kBlockK);
        ok &= encode_kblocked_3d(&maps.a, o.a, o.a_rows, o.lda, kblocks, kBlockM, info.group_kb);
        ok &= encode_kblocked_3d(&maps.b, o.b, o.b_rows, o.ldb, kblocks, bn, info.group_kb);
    } else {
        ok &= encode_2d(&maps.a, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, o.a, k, o.a_rows, o.lda, kBlockK,
                        kBlockM, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B);
        ok &= encode_2d(&maps.b, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, o.b, k, o.b_rows, o.ldb, kBlockK, bn,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B);
    }
    ok &= encode_2d(&maps.d, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, o.d, p.n, o.d_rows, o.ldd * 2, 16,
                    32, CU_TENSOR_MAP_SWIZZLE_32B, CU_TENSOR_MAP_L2_PROMOTION_NONE);
    if (!ok) return DG_ERR_CUDA;
    set_scale_words(p, o);
    p.num_n_blocks = static_cast<int>(cdiv64(p.n, bn));
    p.num_k_blocks = static_cast<int>(cdiv64(k, kBlockK));
    p.group_m = 8;
    p.d = static_cast<uint16_t *>(o.d);
    p.ldd = o.ldd;
    p.timeout_ns = static_cast<uint64_t>(g_timeout_ms.load()) * 1000000ull;
    uint32_t dbg = g_debug_flags.load();
    if (dbg & DG_DEBUG_DROP_ONE_LOAD) g_debug_flags.fetch_and(~static_cast<uint32_t>(DG_DEBUG_DROP_ONE_LOAD));
    p.debug_flags = dbg;
    const int64_t tiles = max_tiles_per_n_block * p.num_n_blocks;
    const int grid = static_cast<int>(tiles < num_sms ? (tiles < 1 ? 1 : tiles) : num_sms);
    if ((dbg & DG_DEBUG_PRINT_CONFIGS) || std::getenv("DG_PRINT_CONFIGS"))
        std::fprintf(stderr, "[dg] mode=%d rows=%d n=%d k=%d -> BLOCK_M=%d BLOCK_N=%d stages=%d smem=%d grid=%d\n",
                     p.mode, p.rows, p.n, k, kBlockM, bn, info.stages, info.smem_bytes, grid);
    g_last_config[0] = kBlockM;
    g_last_config[1] = bn;
    g_last_config[2] = info.stages;
    g_last_config[3] = grid;
    g_last_config[4] = 0;
    g_last_config[5] = 1;
    cudaError_t e = launch_bs_gemm(bn, maps, p, grid, stream);
    return e == cudaSuccess ? DG_OK : DG_ERR_CUDA;
}

// FP32 scales: the two-level promotion kernel.  BLOCK_N must divide 128 so a
// tile's columns share one B block scale.
dg_status launch_promotion(GemmParams &p, const void *a, int64_t lda, const void *b, int64_t ldb,
                           void *d, int64_t ldd, int num_sms, cudaStream_t stream) {
    const int64_t m_blocks = cdiv64(p.rows, kBlockM);
    int bn = 128;
    double best = -1.0;
    for (int cand : {32, 64, 128}) {
        const int64_t nb = cdiv64(p.n, cand);
        const int64_t tiles = m_blocks * nb;
        const int64_t waves = cdiv64(tiles, num_sms);
        const double score = static_cast<double>(tiles) / static_cast<double>(waves * num_sms) *
                             static_cast<double>(p.n) / static_cast<double>(nb * cand) *
                             (cand / (cand + 64.0));
        if (score > best + 1e-9) { best = score; bn = cand; }
    }
    KernelInfo info;
    if (!get_promote_kernel_info(bn, &info)) return DG_ERR_UNSUPPORTED;
    TensorMaps maps;
    std::memset(&maps, 0, sizeof(maps));
    bool ok = true;
    ok &= encode_2d(&maps.a, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, a, p.k, p.rows, lda, kBlockK, kBlockM,
                    CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B);
    ok &= encode_2d(&maps.b, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, b, p.k, p.n, ldb, kBlockK, bn,
                    CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B);
    ok &= encode_2d(&maps.d, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, d, p.n, p.rows, ldd * 2, 16, 32,
                    CU_TENSOR_MAP_SWIZZLE_32B, CU_TENSOR_MAP_L2_PROMOTION_NONE);
    if (!ok) return DG_ERR_CUDA;
    p.num_m_blocks = static_cast<int>(m_blocks);
    p.num_n_blocks = static_cast<int>(cdiv64(p.n, bn));
    p.num_k_blocks = static_cast<int>(cdiv64(p.k, kBlockK));
    p.group_m = 8;
    p.d = static_cast<uint16_t *>(d);
    p.ldd = ldd;
    p.timeout_ns = static_cast<uint64_t>(g_timeout_ms.load()) * 1000000ull;
    p.debug_flags = 0;
    const int64_t tiles = m_blocks * p.num_n_blocks;
    const int grid = static_cast<int>(tiles < num_sms ? tiles : num_sms);
    if (std::getenv("DG_PRINT_CONFIGS") || (g_debug_flags.load() & DG_DEBUG_PRINT_CONFIGS))
        std::fprintf(stderr, "[dg] promote rows=%d n=%d k=%d -> BLOCK_N=%d stages=%d grid=%d\n",
                     p.rows, p.n, p.k, bn, info.stages, grid);
    g_last_config[0] = kBlockM;
    g_last_config[1] = bn;
    g_last_config[2] = info.stages;
    g_last_config[3] = grid;
    g_last_config[4] = 1;
    g_last_config[5] = 1;
    cudaError_t e = launch_promote_gemm(bn, maps, p, grid, stream);
    return e == cudaSuccess ? DG_OK : DG_ERR_CUDA;
}

GemmParams base_params(int mode, int rows, int n, int k, int32_t *status) {
    GemmParams p;
    std::memset(&p, 0, sizeof(p));
    p.mode = mode;
    p.rows = rows;
    p.n = n;
    p.k = k;
    p.num_groups = 1;
    p.status = status;
    p.sf_k = static_cast<int>(cdiv64(k, kGran));
    return p;
}

dg_status check_operand_rules(const void *a, int64_t lda, const void *b, int64_t ldb, int n, int k) {
    if (a == nullptr || b == nullptr) return DG_ERR_INVALID_ARG;
    if (!aligned16(a) || !aligned16(b)) return DG_ERR_ALIGNMENT;
    if (k % 16 != 0 || n % 8 != 0) return DG_ERR_ALIGNMENT;
    if (lda < k || ldb < k) return DG_ERR_INVALID_ARG;
    if (lda % 16 != 0 || ldb % 16 != 0) return DG_ERR_ALIGNMENT;
    return DG_OK;
}

}  // namespace
}  // namespace dg

using namespace dg;

extern "C" {

const char *dg_status_string(int s) {
    switch (s) {
        case DG_OK: return "DG_OK";
        case DG_ERR_INVALID_ARG: return "DG_ERR_INVALID_ARG";
        case DG_ERR_ALIGNMENT: return "DG_ERR_ALIGNMENT";
        case DG_ERR_LAYOUT: return "DG_ERR_LAYOUT";
        case DG_ERR_UNSUPPORTED: return "DG_ERR_UNSUPPORTED";
        case DG_ERR_CUDA: return "DG_ERR_CUDA";
        case DG_ERR_TIMEOUT: return "DG_ERR_TIMEOUT";
        case DG_ERR_INEXACT_SCALE: return "DG_ERR_INEXACT_SCALE";
        case DG_ERR_BAD_GROUP: return "DG_ERR_BAD_GROUP";
        default: return "DG_ERR_UNKNOWN";
    }
}

int dg_get_mk_alignment_for_contiguous_layout(void) { return kBlockM; }

int64_t dg_get_tma_aligned_size(int64_t mn, int elem_size) {
    if (elem_size <= 0 || 16 % elem_size != 0) return -1;
    const int64_t align = 16 / elem_size;
    return (mn + align - 1) / align * align;
}

int64_t dg_packed_sf_words(int batch, int mn, int k) {
    if (batch < 0 || mn < 0 || k < 0) return -1;
    const int64_t sf_k = cdiv64(k, kGran);
    return static_cast<int64_t>(batch) * cdiv64(sf_k, 4) * align4(mn);
}

void dg_set_num_sms(int n) { g_num_sms_override.store(n > 0 ? n : 0); }

int dg_get_num_sms(void) {
    int n = 0;
    if (check_device(&n) != DG_OK) return 0;
    return n;
}

void dg_set_wait_timeout_ms(int ms) { g_timeout_ms.store(ms > 0 ? ms : 2000); }

void dg_set_debug_flags(uint32_t flags) { g_debug_flags.store(flags); }

void dg_get_last_config(int out[6]) {
    for (int i = 0; i < 6; ++i) out[i] = g_last_config[i];
}

dg_status dg_transform_sf(const float *sf, int batch, int mn_rows, int sf_k, int gran_mn, int mn,
                          int out_fmt, void *out, int32_t *status_dev, void *stream) {
    if (batch < 0 || mn < 0 || sf_k < 0 || mn_rows < 0) return DG_ERR_INVALID_ARG;
    if (gran_mn != 1 && gran_mn != kGran) return DG_ERR_UNSUPPORTED;
    if (out_fmt != DG_SF_FP32 && out_fmt != DG_SF_UE8M0_PACKED) return DG_ERR_INVALID_ARG;
    if (static_cast<int64_t>(mn_rows) != cdiv64(mn, gran_mn)) return DG_ERR_LAYOUT;
    if (batch == 0 || mn == 0 || sf_k == 0) return DG_OK;
    if (batch > 65535 || sf_k > 65535 * 4) return DG_ERR_UNSUPPORTED;
    if (sf == nullptr || out == nullptr) return DG_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(sf) & 3u) || !aligned16(out)) return DG_ERR_ALIGNMENT;
    int sms = 0;
    dg_status st = check_device(&sms);
    if (st != DG_OK) return st;
    cudaError_t e = launch_transform_sf(sf, batch, mn_rows, sf_k, gran_mn, mn, out_fmt, out,
                                        status_dev, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? DG_OK : DG_ERR_CUDA;
}

dg_status dg_fp8_gemm_nt(const void *a, int64_t lda, const void *sfa, int sfa_fmt, const void *b,
                         int64_t ldb, const void *sfb, int sfb_fmt, const void *c, int64_t ldc,
                         void *d, int64_t ldd, int m, int n, int k, int32_t *status_dev,
                         void *stream) {
    if (m < 0 || n < 0 || k < 0) return DG_ERR_INVALID_ARG;
    if ((sfa_fmt != DG_SF_FP32 && sfa_fmt != DG_SF_UE8M0_PACKED) ||
        (sfb_fmt != DG_SF_FP32 && sfb_fmt != DG_SF_UE8M0_PACKED))
        return DG_ERR_INVALID_ARG;
    if (sfa_fmt != sfb_fmt) return DG_ERR_UNSUPPORTED;
    if (m == 0 || n == 0) return DG_OK;
    if (d == nullptr) return DG_ERR_INVALID_ARG;
    if (!aligned16(d) || ldd < n || ldd % 8 != 0 || n % 8 != 0) return DG_ERR_ALIGNMENT;
    if (c != nullptr && (!aligned16(c) || ldc < n || ldc % 8 != 0)) return DG_ERR_ALIGNMENT;
    int sms = 0;
    if (k == 0) {
        dg_status st = check_device(&sms);
        if (st != DG_OK) return st;
        dg_fill_d_kernel<<<sms * 4, 256, 0, static_cast<cudaStream_t>(stream)>>>(
            static_cast<const uint16_t *>(c), ldc, static_cast<uint16_t *>(d), ldd, m, n);
        g_last_config[5] = 1;
        return cudaGetLastError() == cudaSuccess ? DG_OK : DG_ERR_CUDA;
    }
    dg_status st = check_operand_rules(a, lda, b, ldb, n, k);
    if (st != DG_OK) return st;
    if (sfa == nullptr || sfb == nullptr) return DG_ERR_INVALID_ARG;
    if (sfa_fmt == DG_SF_UE8M0_PACKED && (!aligned16(sfa) || !aligned16(sfb))) return DG_ERR_ALIGNMENT;
    st = check_device(&sms);
    if (st != DG_OK) return st;
    GemmParams p = base_params(kModeDense, m, n, k, status_dev);
    p.c = static_cast<const uint16_t *>(c);
    p.ldc = ldc;
    if (sfa_fmt == DG_SF_FP32) {
        if (reinterpret_cast<uintptr_t>(sfa) & 3u || reinterpret_cast<uintptr_t>(sfb) & 3u)
            return DG_ERR_ALIGNMENT;
        p.sfa_f32 = static_cast<const float *>(sfa);
        p.sfb_f32 = static_cast<const float *>(sfb);
        return launch_promotion(p, a, lda, b, ldb, d, ldd, sms, static_cast<cudaStream_t>(stream));
    }
    const int64_t psf_k = cdiv64(cdiv64(k, kGran), 4);
    p.num_m_blocks = static_cast<int>(cdiv64(m, kBlockM));
    BsOperands o{a,   lda, static_cast<uint64_t>(m), b,   ldb, static_cast<uint64_t>(n),
                 sfa, static_cast<uint64_t>(m), static_cast<uint64_t>(psf_k),
                 sfb, static_cast<uint64_t>(n), static_cast<uint64_t>(psf_k),
                 d,   ldd, static_cast<uint64_t>(m)};
    return launch_block_scaled(p, o, p.num_m_blocks, p.num_m_blocks, sms,
                               static_cast<cudaStream_t>(stream));
}

dg_status dg_fp8_gemm_nt_f32(const void *a, int64_t lda, const void *sfa, int sfa_fmt, const void *b,
                             int64_t ldb, const void *sfb, int sfb_fmt, const float *c, int64_t ldc,
                             float *d, int64_t ldd, int m, int n, int k, int32_t *status_dev,
                             void *stream) {
    if (m < 0 || n < 0 || k < 0) return DG_ERR_INVALID_ARG;
    if ((sfa_fmt != DG_SF_FP32 && sfa_fmt != DG_SF_UE8M0_PACKED) ||
        (sfb_fmt != DG_SF_FP32 && sfb_fmt != DG_SF_UE8M0_PACKED))
        return DG_ERR_INVALID_ARG;
    if (sfa_fmt != DG_SF_UE8M0_PACKED || sfb_fmt != DG_SF_UE8M0_PACKED) return DG_ERR_UNSUPPORTED;
    if (m == 0 || n == 0) return DG_OK;
    if (d == nullptr) return DG_ERR_INVALID_ARG;
    // FP32 rows: 16-byte aligned starts and 4-column multiples
    if (!aligned16(d) || ldd < n || ldd % 4 != 0 || n % 4 != 0) return DG_ERR_ALIGNMENT;
    if (c != nullptr && (!aligned16(c) || ldc < n || ldc % 4 != 0)) return DG_ERR_ALIGNMENT;
    int sms = 0;
    if (k == 0) {
        dg_status st = check_device(&sms);
        if (st != DG_OK) return st;
        dg_fill_d_f32_kernel<<<sms * 4, 256, 0, static_cast<cudaStream_t>(stream)>>>(c, ldc, d, ldd, m, n);
        g_last_config[5] = 1;
        return cudaGetLastError() == cudaSuccess ? DG_OK : DG_ERR_CUDA;
    }
    dg_status st = check_operand_rules(a, lda, b, ldb, n, k);
    if (st != DG_OK) return st;
    if (sfa == nullptr || sfb == nullptr) return DG_ERR_INVALID_ARG;
    if (!aligned16(sfa) || !aligned16(sfb)) return DG_ERR_ALIGNMENT;
    st = check_device(&sms);
    if (st != DG_OK) return st;
    GemmParams p = base_params(kModeDense, m, n, k, status_dev);
    p.d_f32 = d;
    p.c_f32 = c;
    p.ldc = ldc;
    const int64_t psf_k = cdiv64(cdiv64(k, kGran), 4);
    BsOperands o{a,   lda, static_cast<uint64_t>(m), b,   ldb, static_cast<uint64_t>(n),
                 sfa, static_cast<uint64_t>(m), static_cast<uint64_t>(psf_k),
                 sfb, static_cast<uint64_t>(n), static_cast<uint64_t>(psf_k),
                 d,   ldd, static_cast<uint64_t>(m)};
    // FP32 output runs on 256-row CTA pairs for every M
    const int64_t units = cdiv64(m, 2 * kBlockM);
    return launch_pair(p, o, 256, choose_pair_block_n(p, c != nullptr, units, sms), units, sms,
                       static_cast<cudaStream_t>(stream));
}

// NN / TN / TT: D = C + op(A) op(B) with MN-major operands where the layout
// letter says so; 256x256 CTA-pair tiles.
static dg_status gemm_mn_layout(int lay, const void *a, int64_t lda, const void *sfa, int sfa_fmt,
                                const void *b, int64_t ldb, const void *sfb, int sfb_fmt, const void *c,
                                int64_t ldc, void *d, int64_t ldd, int m, int n, int k, int32_t *status_dev,
                                void *stream) {
    if (m < 0 || n < 0 || k < 0) return DG_ERR_INVALID_ARG;
    if ((sfa_fmt != DG_SF_FP32 && sfa_fmt != DG_SF_UE8M0_PACKED) ||
        (sfb_fmt != DG_SF_FP32 && sfb_fmt != DG_SF_UE8M0_PACKED))
        return DG_ERR_INVALID_ARG;
    if (sfa_fmt != DG_SF_UE8M0_PACKED || sfb_fmt != DG_SF_UE8M0_PACKED) return DG_ERR_UNSUPPORTED;
    if (m == 0 || n == 0) return DG_OK;
    if (d == nullptr) return DG_ERR_INVALID_ARG;
    if (!aligned16(d) || ldd < n || ldd % 8 != 0 || n % 8 != 0) return DG_ERR_ALIGNMENT;
    if (c != nullptr && (!aligned16(c) || ldc < n || ldc % 8 != 0)) return DG_ERR_ALIGNMENT;
    int sms = 0;
    if (k == 0) {
        dg_status st = check_device(&sms);
        if (st != DG_OK) return st;
        dg_fill_d_kernel<<<sms * 4, 256, 0, static_cast<cudaStream_t>(stream)>>>(
            static_cast<const uint16_t *>(c), ldc, static_cast<uint16_t *>(d), ldd, m, n);
        g_last_config[5] = 1;
        return cudaGetLastError() == cudaSuccess ? DG_OK : DG_ERR_CUDA;
    }
    if (a == nullptr || b == nullptr || sfa == nullptr || sfb == nullptr) return DG_ERR_INVALID_ARG;
    if (!aligned16(a) || !aligned16(b) || !aligned16(sfa) || !aligned16(sfb)) return DG_ERR_ALIGNMENT;
    // the contiguous dimension of each operand: K (K-major) or M / N (MN-major)
    const int64_t a_inner = (lay & 1) ? m : k, b_inner = (lay & 2) ? n : k;
    if (lda < a_inner || ldb < b_inner) return DG_ERR_INVALID_ARG;
    if (lda % 16 != 0 || ldb % 16 != 0) return DG_ERR_ALIGNMENT;
    if ((!(lay & 1) || !(lay & 2)) && k % 16 != 0) return DG_ERR_ALIGNMENT;
    dg_status st = check_device(&sms);
    if (st != DG_OK) return st;
    GemmParams p = base_params(kModeDense, m, n, k, status_dev);
    p.c = static_cast<const uint16_t *>(c);
    p.ldc = ldc;
    p.layout = lay;
    const int64_t psf_k = cdiv64(cdiv64(k, kGran), 4);
    BsOperands o{a,   lda, static_cast<uint64_t>(m), b,   ldb, static_cast<uint64_t>(n),
                 sfa, static_cast<uint64_t>(m), static_cast<uint64_t>(psf_k),
                 sfb, static_cast<uint64_t>(n), static_cast<uint64_t>(psf_k),
                 d,   ldd, static_cast<uint64_t>(m)};
    const int64_t units = cdiv64(m, 2 * kBlockM);
    // with C, 224 columns: two TMEM accumulators, so a tile's epilogue overlaps the next one's MMAs
    return launch_pair(p, o, 256, c != nullptr ? 224 : 256, units, sms, static_cast<cudaStream_t>(stream));
}

dg_status dg_fp8_gemm_nn(const void *a, int64_t lda, const void *sfa, int sfa_fmt, const void *b,
                         int64_t ldb, const void *sfb, int sfb_fmt, const void *c, int64_t ldc,
                         void *d, int64_t ldd, int m, int n, int k, int32_t *status_dev, void *stream) {
    return gemm_mn_layout(2, a, lda, sfa, sfa_fmt, b, ldb, sfb, sfb_fmt, c, ldc, d, ldd, m, n, k, status_dev,
                          stream);
}

dg_status dg_fp8_gemm_tn(const void *a, int64_t lda, const void *sfa, int sfa_fmt, const void *b,
                         int64_t ldb, const void *sfb, int sfb_fmt, const void *c, int64_t ldc,
                         void *d, int64_t ldd, int m, int n, int k, int32_t *status_dev, void *stream) {
    return gemm_mn_layout(3, a, lda, sfa, sfa_fmt, b, ldb, sfb, sfb_fmt, c, ldc, d, ldd, m, n, k, status_dev,
                          stream);
}

dg_status dg_fp8_gemm_tt(const void *a, int64_t lda, const void *sfa, int sfa_fmt, const void *b,
                         int64_t ldb, const void *sfb, int sfb_fmt, const void *c, int64_t ldc,
                         void *d, int64_t ldd, int m, int n, int k, int32_t *status_dev, void *stream) {
    return gemm_mn_layout(1, a, lda, sfa, sfa_fmt, b, ldb, sfb, sfb_fmt, c, ldc, d, ldd, m, n, k, status_dev,
                          stream);
}

// FP8 x FP4: 256-row CTA pairs; without C the column count that fills the SMs
// best, of 128 and 256 (one accumulator at 256); with C, 128.
static int choose_fp4_block_n(int64_t m_units, int n, int num_sms, bool with_c) {
    if (with_c) return 128;
    const int cands[2] = {128, 256};
    const int pairs = num_sms / 2;
    double best = -1.0;
    int best_bn = 128;
    for (int bn : cands) {
        const int64_t tiles = m_units * cdiv64(n, bn);
        const int64_t waves = cdiv64(tiles, pairs);
        const double wave_eff = static_cast<double>(tiles) / static_cast<double>(waves * pairs);
        const double pad_eff = static_cast<double>(n) / static_cast<double>(cdiv64(n, bn) * bn);
        const double tile_eff = static_cast<double>(bn) / (bn + 64.0);
        const double score = wave_eff * pad_eff * tile_eff;
        if (score > best + 1e-9) {
            best = score;
            best_bn = bn;
        }
    }
    return best_bn;
}

dg_status dg_fp8_fp4_gemm_nt(const void *a, int64_t lda, const void *sfa, const void *b, int64_t ldb,
                             const void *sfb, const void *c, int64_t ldc, void *d, int64_t ldd, int m, int n,
                             int k, int32_t *status_dev, void *stream) {
    if (m < 0 || n < 0 || k < 0) return DG_ERR_INVALID_ARG;
    if (m == 0 || n == 0) return DG_OK;
    if (d == nullptr) return DG_ERR_INVALID_ARG;
    if (!aligned16(d) || ldd < n || ldd % 8 != 0 || n % 8 != 0) return DG_ERR_ALIGNMENT;
    if (c != nullptr && (!aligned16(c) || ldc < n || ldc % 8 != 0)) return DG_ERR_ALIGNMENT;
    int sms = 0;
    if (k == 0) {
        dg_status st = check_device(&sms);
        if (st != DG_OK) return st;
        dg_fill_d_kernel<<<sms * 4, 256, 0, static_cast<cudaStream_t>(stream)>>>(
            static_cast<const uint16_t *>(c), ldc, static_cast<uint16_t *>(d), ldd, m, n);
        g_last_config[5] = 1;
        return cudaGetLastError() == cudaSuccess ? DG_OK : DG_ERR_CUDA;
    }
    if (a == nullptr || b == nullptr || sfa == nullptr || sfb == nullptr) return DG_ERR_INVALID_ARG;
    if (!aligned16(a) || !aligned16(sfa) || !aligned16(sfb)) return DG_ERR_ALIGNMENT;
    // the FP4 loads: K a multiple of 128, rows 32-byte aligned
    if (k % kBlockK != 0) return DG_ERR_ALIGNMENT;
    if ((reinterpret_cast<uintptr_t>(b) & 31u) != 0 || ldb % 32 != 0) return DG_ERR_ALIGNMENT;
    if (lda < k || ldb < k / 2) return DG_ERR_INVALID_ARG;
    if (lda % 16 != 0) return DG_ERR_ALIGNMENT;
    dg_status st = check_device(&sms);
    if (st != DG_OK) return st;
    GemmParams p = base_params(kModeDense, m, n, k, status_dev);
    p.c = static_cast<const uint16_t *>(c);
    p.ldc = ldc;
    p.layout = 4;
    const int64_t psf_a = cdiv64(cdiv64(k, kGran), 4);   // 4 x 128 K per A word
    const int64_t psf_b = k / kBlockK;                     // 4 x 32 K per B word
    BsOperands o{a,   lda, static_cast<uint64_t>(m), b,   ldb, static_cast<uint64_t>(n),
                 sfa, static_cast<uint64_t>(m), static_cast<uint64_t>(psf_a),
                 sfb, static_cast<uint64_t>(n), static_cast<uint64_t>(psf_b),
                 d,   ldd, static_cast<uint64_t>(m)};
    if (m <= kBlockM && c == nullptr) {
        // M <= 128: 128-row pairs (each CTA loads 64 rows of A), the widest tile that
        // still gives most pairs a tile, as the weight stream from HBM sets the time
        int bn = 32;
        for (int cand : {128, 96})
            if (cdiv64(n, cand) * 10 >= static_cast<int64_t>(sms / 2) * 9) {
                bn = cand;
                break;
            }
        return launch_pair(p, o, 128, bn, 1, sms, static_cast<cudaStream_t>(stream));
    }
    const int64_t units = cdiv64(m, 2 * kBlockM);
    const int bn = choose_fp4_block_n(units, n, sms, c != nullptr);
    return launch_pair(p, o, 256, bn, units, sms, static_cast<cudaStream_t>(stream));
}

// Operand rules of the FP4 weights: K a multiple of 128, rows 32-byte aligned.
static dg_status check_fp4_operands(const void *a, int64_t lda, const void *b, int64_t ldb, int n, int k) {
    if (a == nullptr || b == nullptr) return DG_ERR_INVALID_ARG;
    if (!aligned16(a) || (reinterpret_cast<uintptr_t>(b) & 31u) != 0) return DG_ERR_ALIGNMENT;
    if (k % kBlockK != 0 || n % 8 != 0 || ldb % 32 != 0 || lda % 16 != 0) return DG_ERR_ALIGNMENT;
    if (lda < k || ldb < k / 2) return DG_ERR_INVALID_ARG;
    return DG_OK;
}

dg_status dg_m_grouped_fp8_fp4_gemm_nt_contiguous(const void *a, int64_t lda, const void *sfa, const void *b,
                                                  int64_t ldb, const void *sfb, void *d, int64_t ldd,
                                                  const int32_t *grouped_layout, int m_total, int n, int k,
                                                  int num_groups, int32_t *status_dev, void *stream) {
    if (m_total < 0 || n < 0 || k < 0 || num_groups < 1) return DG_ERR_INVALID_ARG;
    if (m_total % kBlockM != 0) return DG_ERR_LAYOUT;
    if (m_total == 0 || n == 0) return DG_OK;
    if (k == 0) return DG_ERR_UNSUPPORTED;
    dg_status st = check_fp4_operands(a, lda, b, ldb, n, k);
    if (st != DG_OK) return st;
    if (d == nullptr || sfa == nullptr || sfb == nullptr || grouped_layout == nullptr) return DG_ERR_INVALID_ARG;
    if (!aligned16(d) || !aligned16(sfa) || !aligned16(sfb) || ldd < n || ldd % 8 != 0) return DG_ERR_ALIGNMENT;
    if (static_cast<int64_t>(num_groups) * n > INT32_MAX || cdiv64(m_total, 2 * kBlockM) > kMaxPairPrefix ||
        num_groups >= 32768)
        return DG_ERR_UNSUPPORTED;
    int sms = 0;
    st = check_device(&sms);
    if (st != DG_OK) return st;
    GemmParams p = base_params(kModeContiguous, m_total, n, k, status_dev);
    p.num_groups = num_groups;
    p.grouped_layout = grouped_layout;
    p.layout = 4;
    const int64_t psf_a = cdiv64(cdiv64(k, kGran), 4);
    const int64_t kb = k / kBlockK;
    BsOperands o{a,   lda, static_cast<uint64_t>(m_total),
                 b,   ldb, static_cast<uint64_t>(num_groups) * n,
                 sfa, static_cast<uint64_t>(m_total), static_cast<uint64_t>(psf_a),
                 sfb, static_cast<uint64_t>(n), static_cast<uint64_t>(kb * num_groups),
                 d,   ldd, static_cast<uint64_t>(m_total)};
    const int64_t blocks = m_total / kBlockM;
    const int bn = choose_fp4_block_n(cdiv64(blocks, 2), n, sms, false);
    return launch_pair(p, o, 256, bn, blocks, sms, static_cast<cudaStream_t>(stream));
}

dg_status dg_m_grouped_fp8_fp4_gemm_nt_masked(const void *a, const void *sfa, const void *b, const void *sfb,
                                              void *d, const int32_t *masked_m, int num_groups, int max_m,
                                              int expected_m, int n, int k, int32_t *status_dev, void *stream) {
    if (num_groups < 1 || max_m < 0 || n < 0 || k < 0) return DG_ERR_INVALID_ARG;
    if (num_groups > kMaxPairPrefix) return DG_ERR_UNSUPPORTED;
    if (max_m == 0 || n == 0) return DG_OK;
    if (k == 0) return DG_ERR_UNSUPPORTED;
    dg_status st = check_fp4_operands(a, k, b, k / 2, n, k);
    if (st != DG_OK) return st;
    if (d == nullptr || sfa == nullptr || sfb == nullptr || masked_m == nullptr) return DG_ERR_INVALID_ARG;
    if (!aligned16(d) || !aligned16(sfa) || !aligned16(sfb)) return DG_ERR_ALIGNMENT;
    if (static_cast<int64_t>(num_groups) * max_m > INT32_MAX || static_cast<int64_t>(num_groups) * n > INT32_MAX)
        return DG_ERR_UNSUPPORTED;
    int sms = 0;
    st = check_device(&sms);
    if (st != DG_OK) return st;
    GemmParams p = base_params(kModeMasked, max_m, n, k, status_dev);
    p.num_groups = num_groups;
    p.masked_m = masked_m;
    p.layout = 4;
    p.num_m_blocks = static_cast<int>(cdiv64(max_m, kBlockM));
    const int64_t psf_a = cdiv64(cdiv64(k, kGran), 4);
    const int64_t kb = k / kBlockK;
    BsOperands o{a,   k,     static_cast<uint64_t>(num_groups) * max_m,
                 b,   k / 2, static_cast<uint64_t>(num_groups) * n,
                 sfa, static_cast<uint64_t>(max_m), static_cast<uint64_t>(psf_a * num_groups),
                 sfb, static_cast<uint64_t>(n), static_cast<uint64_t>(kb * num_groups),
                 d,   n,     static_cast<uint64_t>(num_groups) * max_m};
    const int exp_m = expected_m > 0 ? (expected_m < max_m ? expected_m : max_m) : max_m;
    const int bn = choose_fp4_block_n(static_cast<int64_t>(num_groups) * cdiv64(exp_m, 2 * kBlockM), n, sms, false);
    return launch_pair(p, o, 256, bn, static_cast<int64_t>(num_groups) * p.num_m_blocks, sms,
                       static_cast<cudaStream_t>(stream));
}

dg_status dg_m_grouped_fp8_gemm_nt_contiguous(const void *a, int64_t lda, const void *sfa,
                                              int sfa_fmt, const void *b, int64_t ldb,
                                              const void *sfb, int sfb_fmt, void *d, int64_t ldd,
                                              const int32_t *grouped_layout, int m_total, int n,
                                              int k, int num_groups, int32_t *status_dev,
                                              void *stream) {
    if (m_total < 0 || n < 0 || k < 0 || num_groups < 1) return DG_ERR_INVALID_ARG;
    if ((sfa_fmt != DG_SF_FP32 && sfa_fmt != DG_SF_UE8M0_PACKED) ||
        (sfb_fmt != DG_SF_FP32 && sfb_fmt != DG_SF_UE8M0_PACKED))
        return DG_ERR_INVALID_ARG;
    if (sfa_fmt != DG_SF_UE8M0_PACKED || sfb_fmt != DG_SF_UE8M0_PACKED) return DG_ERR_UNSUPPORTED;
    if (m_total % kBlockM != 0) return DG_ERR_LAYOUT;
    if (m_total == 0 || n == 0) return DG_OK;
    if (k == 0) return DG_ERR_UNSUPPORTED;
    dg_status st = check_operand_rules(a, lda, b, ldb, n, k);
    if (st != DG_OK) return st;
    if (d == nullptr || sfa == nullptr || sfb == nullptr || grouped_layout == nullptr)
        return DG_ERR_INVALID_ARG;
    if (!aligned16(d) || !aligned16(sfa) || !aligned16(sfb) || ldd < n || ldd % 8 != 0)
        return DG_ERR_ALIGNMENT;
    if (static_cast<int64_t>(num_groups) * n > INT32_MAX) return DG_ERR_UNSUPPORTED;
    int sms = 0;
    st = check_device(&sms);
    if (st != DG_OK) return st;
    GemmParams p = base_params(kModeContiguous, m_total, n, k, status_dev);
    p.num_groups = num_groups;
    p.grouped_layout = grouped_layout;
    p.num_m_blocks = m_total / kBlockM;
    const int64_t psf_k = cdiv64(cdiv64(k, kGran), 4);
    BsOperands o{a,   lda, static_cast<uint64_t>(m_total),
                 b,   ldb, static_cast<uint64_t>(num_groups) * n,
                 sfa, static_cast<uint64_t>(m_total), static_cast<uint64_t>(psf_k),
                 sfb, static_cast<uint64_t>(n), static_cast<uint64_t>(psf_k * num_groups),
                 d,   ldd, static_cast<uint64_t>(m_total)};
    return launch_block_scaled(p, o, p.num_m_blocks, p.num_m_blocks, sms,
                               static_cast<cudaStream_t>(stream));
}

dg_status dg_m_grouped_fp8_gemm_nt_contiguous_psum(const void *a, int64_t lda, const void *sfa,
                                                   int sfa_fmt, const void *b, int64_t ldb,
                                                   const void *sfb, int sfb_fmt, void *d, int64_t ldd,
                                                   const int32_t *psum, int m_total, int n, int k,
                                                   int num_groups, int32_t *status_dev, void *stream) {
    if (m_total < 0 || n < 0 || k < 0 || num_groups < 1) return DG_ERR_INVALID_ARG;
    if ((sfa_fmt != DG_SF_FP32 && sfa_fmt != DG_SF_UE8M0_PACKED) ||
        (sfb_fmt != DG_SF_FP32 && sfb_fmt != DG_SF_UE8M0_PACKED))
        return DG_ERR_INVALID_ARG;
    if (sfa_fmt != DG_SF_UE8M0_PACKED || sfb_fmt != DG_SF_UE8M0_PACKED) return DG_ERR_UNSUPPORTED;
    if (m_total % kBlockM != 0) return DG_ERR_LAYOUT;
    // the PSUM layout runs on 256-row CTA pairs only
    if (num_groups > kMaxPsumGroups || cdiv64(m_total, 2 * kBlockM) > kMaxPairPrefix) return DG_ERR_UNSUPPORTED;
    if (m_total == 0 || n == 0) return DG_OK;
    if (k == 0) return DG_ERR_UNSUPPORTED;
    dg_status st = check_operand_rules(a, lda, b, ldb, n, k);
    if (st != DG_OK) return st;
    if (d == nullptr || sfa == nullptr || sfb == nullptr || psum == nullptr) return DG_ERR_INVALID_ARG;
    if (!aligned16(d) || !aligned16(sfa) || !aligned16(sfb) || ldd < n || ldd % 8 != 0)
        return DG_ERR_ALIGNMENT;
    if (static_cast<int64_t>(num_groups) * n > INT32_MAX) return DG_ERR_UNSUPPORTED;
    int sms = 0;
    st = check_device(&sms);
    if (st != DG_OK) return st;
    GemmParams p = base_params(kModeContiguous, m_total, n, k, status_dev);
    p.num_groups = num_groups;
    p.psum = psum;
    p.num_m_blocks = m_total / kBlockM;
    const int64_t psf_k = cdiv64(cdiv64(k, kGran), 4);
    BsOperands o{a,   lda, static_cast<uint64_t>(m_total),
                 b,   ldb, static_cast<uint64_t>(num_groups) * n,
                 sfa, static_cast<uint64_t>(m_total), static_cast<uint64_t>(psf_k),
                 sfb, static_cast<uint64_t>(n), static_cast<uint64_t>(psf_k * num_groups),
                 d,   ldd, static_cast<uint64_t>(m_total)};
    const int64_t units_hint = cdiv64(p.num_m_blocks, 2);
    return launch_pair(p, o, 256, choose_pair_block_n(p, false, units_hint, sms), p.num_m_blocks, sms,
                       static_cast<cudaStream_t>(stream));
}

dg_status dg_m_grouped_fp8_gemm_nt_masked(const void *a, const void *sfa, int sfa_fmt,
                                          const void *b, const void *sfb, int sfb_fmt, void *d,
                                          const int32_t *masked_m, int num_groups, int max_m,
                                          int expected_m, int n, int k, int32_t *status_dev,
                                          void *stream) {
    if (num_groups < 1 || max_m < 0 || n < 0 || k < 0) return DG_ERR_INVALID_ARG;
    if (num_groups > kMaxGroupsMasked) return DG_ERR_UNSUPPORTED;
    if ((sfa_fmt != DG_SF_FP32 && sfa_fmt != DG_SF_UE8M0_PACKED) ||
        (sfb_fmt != DG_SF_FP32 && sfb_fmt != DG_SF_UE8M0_PACKED))
        return DG_ERR_INVALID_ARG;
    if (sfa_fmt != DG_SF_UE8M0_PACKED || sfb_fmt != DG_SF_UE8M0_PACKED) return DG_ERR_UNSUPPORTED;
    if (max_m == 0 || n == 0) return DG_OK;
    if (k == 0) return DG_ERR_UNSUPPORTED;
    dg_status st = check_operand_rules(a, k, b, k, n, k);
    if (st != DG_OK) return st;
    if (d == nullptr || sfa == nullptr || sfb == nullptr || masked_m == nullptr)
        return DG_ERR_INVALID_ARG;
    if (!aligned16(d) || !aligned16(sfa) || !aligned16(sfb)) return DG_ERR_ALIGNMENT;
    if (static_cast<int64_t>(num_groups) * max_m > INT32_MAX ||
        static_cast<int64_t>(num_groups) * n > INT32_MAX)
        return DG_ERR_UNSUPPORTED;
    int sms = 0;
    st = check_device(&sms);
    if (st != DG_OK) return st;
    GemmParams p = base_params(kModeMasked, max_m, n, k, status_dev);
    p.num_groups = num_groups;
    p.masked_m = masked_m;
    p.num_m_blocks = static_cast<int>(cdiv64(max_m, kBlockM));
    const int64_t psf_k = cdiv64(cdiv64(k, kGran), 4);
    const int exp_m = expected_m > 0 ? (expected_m < max_m ? expected_m : max_m) : max_m;
    const int64_t m_blocks_hint = static_cast<int64_t>(num_groups) * cdiv64(exp_m, kBlockM);
    BsOperands o{a,   k,   static_cast<uint64_t>(num_groups) * max_m,
                 b,   k,   static_cast<uint64_t>(num_groups) * n,
                 sfa, static_cast<uint64_t>(max_m), static_cast<uint64_t>(psf_k * num_groups),
                 sfb, static_cast<uint64_t>(n), static_cast<uint64_t>(psf_k * num_groups),
                 d,   n,   static_cast<uint64_t>(num_groups) * max_m};
    return launch_block_scaled(p, o, m_blocks_hint,
                               static_cast<int64_t>(num_groups) * p.num_m_blocks, sms,
                               static_cast<cudaStream_t>(stream));
}

// ------------------------------------------------------------ K-grouped (weight gradient)

// Packed rows of the K-grouped scales (sum of ceil(ks[e] / 512)), or -1 if ks
// is invalid: null with groups, more than 255 groups, a size negative or not a
// multiple of 128, or more than 65535 packed rows.
// Scale rows of the K-grouped layout with one FP32 scale row per gran_k rows of K
// (128, or 32 for the pre-packed form): each group's rows are packed on their
// own, 4 per word.  Returns the packed rows, or -1 for invalid sizes.
static int64_t k_grouped_rows(const int *ks, int num_groups, KGroupRows *t, int gran_k = kBlockK) {
    if (num_groups < 0 || num_groups > kMaxPsumGroups || (num_groups > 0 && ks == nullptr)) return -1;
    int64_t srow = 0, prow = 0;
    if (t) t->num_groups = num_groups;
    for (int e = 0; e < num_groups; ++e) {
        if (ks[e] < 0 || ks[e] % kBlockK != 0) return -1;
        if (t) {
            t->srow[e] = static_cast<int>(srow);
            t->prow[e] = static_cast<int>(prow);
        }
        srow += ks[e] / gran_k;
        prow += (ks[e] / gran_k + 3) / 4;
        if (prow > 65535) return -1;
    }
    if (t) {
        t->srow[num_groups] = static_cast<int>(srow);
        t->prow[num_groups] = static_cast<int>(prow);
    }
    return prow;
}

int64_t dg_k_grouped_packed_sf_rows(const int *ks, int num_groups) {
    return k_grouped_rows(ks, num_groups, nullptr);
}

static dg_status transform_sf_k_grouped(const float *sf, int mn, const int *ks, int num_groups, void *out,
                                        int32_t *status_dev, void *stream, int gran_k) {
    if (mn < 0) return DG_ERR_INVALID_ARG;
    KGroupRows t;
    const int64_t prows = k_grouped_rows(ks, num_groups, &t, gran_k);
    if (prows < 0) return DG_ERR_INVALID_ARG;
    if (mn % 4 != 0) return DG_ERR_LAYOUT;
    if (mn == 0 || prows == 0) return DG_OK;
    if (sf == nullptr || out == nullptr) return DG_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(sf) & 3u) || !aligned16(out)) return DG_ERR_ALIGNMENT;
    int sms = 0;
    dg_status st = check_device(&sms);
    if (st != DG_OK) return st;
    cudaError_t e = launch_transform_sf_k_grouped(sf, mn, t, static_cast<int>(prows), out, status_dev,
                                                  static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? DG_OK : DG_ERR_CUDA;
}

dg_status dg_transform_sf_k_grouped(const float *sf, int mn, const int *ks, int num_groups, void *out,
                                    int32_t *status_dev, void *stream) {
    return transform_sf_k_grouped(sf, mn, ks, num_groups, out, status_dev, stream, kBlockK);
}

dg_status dg_transform_sf_k_grouped_k32(const float *sf, int mn, const int *ks, int num_groups, void *out,
                                        int32_t *status_dev, void *stream) {
    return transform_sf_k_grouped(sf, mn, ks, num_groups, out, status_dev, stream, 32);
}

// The K-grouped GEMM with scales every 128 (k32 false) or 32 (k32 true) rows of K.
static dg_status k_grouped_gemm(const void *a, int64_t lda, const void *sfa, const void *b, int64_t ldb,
                                const void *sfb, const float *c, float *d, int m, int n, const int *ks,
                                const int32_t *ks_dev, int num_groups, int32_t *status_dev, void *stream, bool k32) {
    if (m < 0 || n < 0) return DG_ERR_INVALID_ARG;
    const int64_t prows = k_grouped_rows(ks, num_groups, nullptr, k32 ? 32 : kBlockK);
    if (prows < 0) return DG_ERR_INVALID_ARG;
    if (m == 0 || n == 0 || num_groups == 0) return DG_OK;
    if (c == nullptr || d == nullptr) return DG_ERR_INVALID_ARG;   // C is required
    if (m % 4 != 0 || n % 4 != 0) return DG_ERR_LAYOUT;            // packed scales: mn % 4 == 0
    if (!aligned16(c) || !aligned16(d)) return DG_ERR_ALIGNMENT;
    const int64_t rows = static_cast<int64_t>(num_groups) * m;
    if (rows > INT32_MAX || rows * n > (int64_t(1) << 40)) return DG_ERR_UNSUPPORTED;
    int64_t k_total = 0;
    for (int e = 0; e < num_groups; ++e) k_total += ks[e];
    if (k_total > INT32_MAX) return DG_ERR_UNSUPPORTED;
    int sms = 0;
    dg_status st = check_device(&sms);
    if (st != DG_OK) return st;
    if (k_total == 0) {
        // every group is empty: D = C
        dg_fill_d_f32_kernel<<<sms * 4, 256, 0, static_cast<cudaStream_t>(stream)>>>(c, n, d, n,
                                                                                      static_cast<int>(rows), n);
        g_last_config[5] = 1;
        return cudaGetLastError() == cudaSuccess ? DG_OK : DG_ERR_CUDA;
    }
    if (a == nullptr || b == nullptr || sfa == nullptr || sfb == nullptr || ks_dev == nullptr)
        return DG_ERR_INVALID_ARG;
    if (!aligned16(a) || !aligned16(b) || !aligned16(sfa) || !aligned16(sfb)) return DG_ERR_ALIGNMENT;
    if (lda < m || ldb < n) return DG_ERR_INVALID_ARG;
    if (lda % 16 != 0 || ldb % 16 != 0) return DG_ERR_ALIGNMENT;
    GemmParams p = base_params(kModeKGrouped, static_cast<int>(rows), n, static_cast<int>(k_total), status_dev);
    p.num_groups = num_groups;
    p.ks = ks_dev;
    p.group_rows = m;
    p.num_m_blocks = static_cast<int>(cdiv64(m, 2 * kBlockM));   // m-units of one group
    // A [K][M], B [K][N]; 32-K scales (layout bit 3) take 192-column tiles, the widest
    // whose two accumulators fit beside their four-times-larger TMEM scale slots
    p.layout = k32 ? 3 | 8 : 3;
    p.c_f32 = c;
    p.d_f32 = d;
    p.ldc = n;
    BsOperands o{a,   lda, static_cast<uint64_t>(m), b,   ldb, static_cast<uint64_t>(n),
                 sfa, static_cast<uint64_t>(m), static_cast<uint64_t>(prows),
                 sfb, static_cast<uint64_t>(n), static_cast<uint64_t>(prows),
                 d,   n,   static_cast<uint64_t>(rows)};
    const int64_t units = static_cast<int64_t>(num_groups) * p.num_m_blocks;
    return launch_pair(p, o, 256, k32 ? 192 : 224, units, sms, static_cast<cudaStream_t>(stream));
}

dg_status dg_k_grouped_fp8_gemm_tn_contiguous(const void *a, int64_t lda, const void *sfa, const void *b,
                                              int64_t ldb, const void *sfb, const float *c, float *d, int m,
                                              int n, const int *ks, const int32_t *ks_dev, int num_groups,
                                              int32_t *status_dev, void *stream) {
    return k_grouped_gemm(a, lda, sfa, b, ldb, sfb, c, d, m, n, ks, ks_dev, num_groups, status_dev, stream, false);
}

dg_status dg_k_grouped_fp8_gemm_tn_contiguous_k32(const void *a, int64_t lda, const void *sfa, const void *b,
                                                  int64_t ldb, const void *sfb, const float *c, float *d, int m,
                                                  int n, const int *ks, const int32_t *ks_dev, int num_groups,
                                                  int32_t *status_dev, void *stream) {
    return k_grouped_gemm(a, lda, sfa, b, ldb, sfb, c, d, m, n, ks, ks_dev, num_groups, status_dev, stream, true);
}

}  // extern "C"
