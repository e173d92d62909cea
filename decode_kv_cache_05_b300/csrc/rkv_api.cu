// librkv: C ABI entry points (declared in include/rkv.h). Host-side argument
// validation, tensor-map encoding and kernel launches on the caller's stream.
// No entry point allocates device memory or synchronises the host, except
// rkv_device_status.
#include "rkv.h"

#include <cudaTypedefs.h>

#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "rkv_compact.cuh"
#include "rkv_freelist.cuh"
#include "rkv_importance.cuh"
#include "rkv_redundancy.cuh"
#include "rkv_redundancy_closed.cuh"
#include "rkv_select.cuh"
#include "rkv_select_compact.cuh"

namespace {

using namespace rkv;


// Per-device values that the launchers look up once and then reuse. Several
// host threads may call the library at once: every cache slot is an atomic
// int (0 = not looked up yet); two threads that miss together both look the
// value up and store the same result.
constexpr int kMaxDevices = 64;

// Streaming multiprocessors of the current device (cached per device).
int sm_count()
{
    static std::atomic<int> cached[kMaxDevices];
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0)
        return 0;
    if (dev < kMaxDevices) {
        const int c = cached[dev].load(std::memory_order_relaxed);
        if (c > 0)
            return c;
    }
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return 0;
    if (dev < kMaxDevices)
        cached[dev].store(n, std::memory_order_relaxed);
    return n;
}

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

inline int ceil_div(long long a, long long b) { return static_cast<int>((a + b - 1) / b); }

inline uint32_t pow2_at_least(uint32_t x)
{
    uint32_t p = 32;
    while (p < x)
        p <<= 1;
    return p;
}

rkv_status check_problem(const rkv_problem *p)
{
    if (!p)
        return RKV_ERR_INVALID_ARG;
    if (p->num_layers < 0 || p->batch < 0 || p->num_kv_heads < 1 || p->num_q_heads < 1 || p->budget < 1 ||
        p->window < 1 || p->max_seq_len < 1)
        return RKV_ERR_INVALID_ARG;
    if (p->num_q_heads % p->num_kv_heads != 0 || p->window > p->budget || !std::isfinite(p->mix_lambda))
        return RKV_ERR_INVALID_ARG;
    if (p->layout != RKV_LAYOUT_CONTIGUOUS && p->layout != RKV_LAYOUT_PAGED)
        return RKV_ERR_INVALID_ARG;
    if (p->redundancy != RKV_REDUNDANCY_GRAM && p->redundancy != RKV_REDUNDANCY_CLOSED_FORM &&
        p->redundancy != RKV_REDUNDANCY_CLOSED_FORM_FUSED)
        return RKV_ERR_INVALID_ARG;
    if (p->selection != RKV_SELECT_PER_HEAD && p->selection != RKV_SELECT_SHARED_HEADS)
        return RKV_ERR_INVALID_ARG;
    if (p->trigger != RKV_TRIGGER_ANY && p->trigger != RKV_TRIGGER_BUDGET_PLUS_BUFFER)
        return RKV_ERR_INVALID_ARG;
    if (p->buffer < 0)
        return RKV_ERR_INVALID_ARG;
    if (p->head_dim != kHeadDim || p->max_seq_len > kMaxSeq)
        return RKV_ERR_UNSUPPORTED;
    if ((p->num_q_heads / p->num_kv_heads) * p->window > 64)
        return RKV_ERR_UNSUPPORTED;
    if (p->layout == RKV_LAYOUT_PAGED) {
        if (p->block_size != kBlock)
            return RKV_ERR_UNSUPPORTED;
        if (p->num_blocks < 1 || p->max_blocks_per_seq < ceil_div(p->max_seq_len, kBlock))
            return RKV_ERR_INVALID_ARG;
    }
    const long long heads = static_cast<long long>(p->num_layers) * p->batch * p->num_kv_heads;
    if (heads * 8 > 0x7FFFFFFFll)
        return RKV_ERR_UNSUPPORTED;
    if (heads * p->max_seq_len > 0x7FFFFFFFll)
        return RKV_ERR_UNSUPPORTED; // TMA row coordinates are int32
    return RKV_OK;
}

Geom make_geom(const rkv_problem *p, const int32_t *seq_lens, const int32_t *block_table)
{
    Geom g;
    g.L = p->num_layers;
    g.B = p->batch;
    g.Hkv = p->num_kv_heads;
    g.Hq = p->num_q_heads;
    g.G = p->num_q_heads / p->num_kv_heads;
    g.w = p->window;
    g.rows = g.G * g.w;
    g.nmax = p->max_seq_len;
    g.npad = ceil_div(p->max_seq_len, kTileKeys) * kTileKeys;
    g.paged = p->layout == RKV_LAYOUT_PAGED;
    g.max_blocks = g.paged ? p->max_blocks_per_seq : 0;
    g.num_blocks = g.paged ? p->num_blocks : 0;
    g.budget = p->budget;
    g.lam = p->mix_lambda;
    g.redundancy = p->redundancy;
    g.shared_sel = p->selection == RKV_SELECT_SHARED_HEADS;
    g.buffer = p->buffer;
    g.trigger_at_full = p->trigger == RKV_TRIGGER_BUDGET_PLUS_BUFFER;
    g.seq_lens = seq_lens;
    g.block_table = g.paged ? block_table : nullptr;
    return g;
}

inline long long num_heads(const Geom &g) { return static_cast<long long>(g.L) * g.B * g.Hkv; }

// A driver entry point by name (nullptr if the driver lacks it).
void *driver_entry(const char *name, int version)
{
    void *ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion(name, &ptr, version, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
        return nullptr;
    return ptr;
}

// The function-local static is initialised once, by whichever thread comes
// first (C++11 guarantees the others wait for it).
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder()
{
    static const auto fn =
        reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(driver_entry("cuTensorMapEncodeTiled", 12000));
    return fn;
}

// K (or V) as TMA sees it: 128-row x 64-column boxes (contiguous) or 16-row
// boxes of one head inside one pool block (paged), 128-byte swizzle.
bool encode_k_map(CUtensorMap *map, const Geom &g, const void *k)
{
    auto enc = tensor_map_encoder();
    if (!enc)
        return false;
    CUresult r;
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    if (!g.paged) {
        const cuuint64_t dims[2] = {static_cast<cuuint64_t>(kHeadDim),
                                    static_cast<cuuint64_t>(num_heads(g)) * g.nmax};
        const cuuint64_t strides[1] = {kHeadDim * 2};
        const cuuint32_t box[2] = {64, kTileKeys};
        r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(k), dims, strides, box, estr,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    } else {
        const cuuint64_t dims[4] = {static_cast<cuuint64_t>(kHeadDim), static_cast<cuuint64_t>(g.Hkv),
                                    static_cast<cuuint64_t>(kBlock),
                                    static_cast<cuuint64_t>(g.L) * g.num_blocks};
        const cuuint64_t row = kHeadDim * 2;
        const cuuint64_t strides[3] = {row, row * g.Hkv, row * g.Hkv * kBlock};
        const cuuint32_t box[4] = {64, 1, kBlock, 1};
        r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(k), dims, strides, box, estr,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    }
    return r == CUDA_SUCCESS;
}

// Key rows without swizzle (256 contiguous bytes per row in shared memory):
// boxes of `rows` rows on the contiguous layout, of one 16-token block on the
// paged one.
bool encode_k_rows_map(CUtensorMap *map, const Geom &g, const void *k, int rows)
{
    auto enc = tensor_map_encoder();
    if (!enc)
        return false;
    CUresult r;
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    if (!g.paged) {
        const cuuint64_t dims[2] = {static_cast<cuuint64_t>(kHeadDim),
                                    static_cast<cuuint64_t>(num_heads(g)) * g.nmax};
        const cuuint64_t strides[1] = {kHeadDim * 2};
        const cuuint32_t box[2] = {kHeadDim, static_cast<cuuint32_t>(rows)};
        r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(k), dims, strides, box, estr,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    } else {
        const cuuint64_t dims[4] = {static_cast<cuuint64_t>(kHeadDim), static_cast<cuuint64_t>(g.Hkv),
                                    static_cast<cuuint64_t>(kBlock),
                                    static_cast<cuuint64_t>(g.L) * g.num_blocks};
        const cuuint64_t row = kHeadDim * 2;
        const cuuint64_t strides[3] = {row, row * g.Hkv, row * g.Hkv * kBlock};
        const cuuint32_t box[4] = {kHeadDim, 1, kBlock, 1};
        r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(k), dims, strides, box, estr,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    }
    return r == CUDA_SUCCESS;
}

bool encode_q_map(CUtensorMap *map, const Geom &g, const void *q, int nr)
{
    auto enc = tensor_map_encoder();
    if (!enc)
        return false;
    const cuuint32_t estr[2] = {1, 1};
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(kHeadDim),
                                static_cast<cuuint64_t>(g.L) * g.B * g.Hq * g.w};
    const cuuint64_t strides[1] = {kHeadDim * 2};
    const cuuint32_t box[2] = {64, static_cast<cuuint32_t>(nr)};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(q), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Programmatic dependent launch (the next kernel in the stream scheduled
// while this one drains; the kernels run their set-up, then wait in
// griddepcontrol.wait). 0: never; 1: always; 2 (default): for problems with
// fewer heads than SMs only. Measured on B300, every kernel in plain stream
// order gave the Llama-3-8B cache 218,684 -> 221,249 events/s, the paged
// Qwen2-7B cache 432,650 -> 453,346, Llama-8B at B = 64 87,282 -> 95,130 and
// its closed form 174,808 -> 193,493 -- the early-scheduled CTAs of the next
// kernel (a persistent redundancy grid, or select + compact after one)
// started skewed against their fixed shares of the work -- while the
// one-layer case (8 heads, one short wave per kernel) lost 26,072 -> 24,692.
#ifndef RKV_PDL
#define RKV_PDL 2
#endif
// Whether the launches of the current entry-point call may use it (RKV_PDL
// 2), set per call and per host thread by PdlScope.
thread_local bool t_small_problem = false;

// Raises a kernel's dynamic shared-memory limit once per (kernel, device): a
// repeat call, such as one recorded into a CUDA graph after a first eager
// call, then issues no attribute change.
bool ensure_smem_limit(const void *func, size_t smem)
{
    if (smem <= 48 * 1024)
        return true;
    struct Entry {
        const void *func;
        int dev;
        size_t smem;
    };
    static Entry entries[256];
    static int count = 0;
    static std::mutex mu;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess)
        return false;
    std::lock_guard<std::mutex> lock(mu);
    for (int i = 0; i < count; ++i)
        if (entries[i].func == func && entries[i].dev == dev && entries[i].smem >= smem)
            return true;
    if (cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)) !=
        cudaSuccess)
        return false;
    if (count < 256)
        entries[count++] = Entry{func, dev, smem};
    return true;
}

template <typename Kernel, typename... Args>
rkv_status launch(Kernel kernel, dim3 grid, dim3 block, size_t smem, int cluster, cudaStream_t stream,
                  Args... args)
{
    if (!ensure_smem_limit(reinterpret_cast<const void *>(kernel), smem))
        return RKV_ERR_CUDA;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(cluster);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    // programmatic dependent launch: the kernel may be scheduled while the
    // previous kernel in the stream drains; it runs its set-up (barriers,
    // TMEM) and then waits in griddepcontrol.wait before touching memory
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = RKV_PDL == 1 || (RKV_PDL == 2 && t_small_problem);
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    if (cudaLaunchKernelEx(&cfg, kernel, args...) != cudaSuccess)
        return RKV_ERR_CUDA;
    return RKV_OK;
}

struct ImpPlan {
    int nr, cluster, tiles_per_cta, stages;
    uint32_t tmem_cols;
};

// At most this many 128-key tiles per importance CTA (a cluster of CTAs
// splits longer heads). Measured on B300: smaller clusters cost less in
// cross-CTA softmax exchanges; eight tiles of 32 logit columns still let two
// CTAs share an SM's TMEM.
#ifndef RKV_IMP_MAX_TILES
#define RKV_IMP_MAX_TILES 8
#endif

ImpPlan plan_importance(const Geom &g)
{
    ImpPlan pl;
    pl.nr = g.rows <= 32 ? 32 : 64;
    const int tiles_max = ceil_div(g.nmax, kTileKeys);
    const int c = ceil_div(tiles_max, std::min(RKV_IMP_MAX_TILES, kImpMaxTiles));
    pl.tiles_per_cta = ceil_div(tiles_max, c);
    pl.cluster = ceil_div(tiles_max, pl.tiles_per_cta);
    pl.tmem_cols = pow2_at_least(static_cast<uint32_t>(pl.tiles_per_cta * pl.nr));
    // A ring as deep as the CTA's tiles, limited so that two CTAs still fit an
    // SM's shared memory when TMEM allows more than one.
    const int smem_cap = pl.tmem_cols > 256 ? 4 : (pl.nr == 32 ? 3 : 2);
    pl.stages = std::max(2, std::min(pl.tiles_per_cta, smem_cap));
    return pl;
}

template <int NR>
rkv_status launch_importance(const ImpPlan &pl, dim3 grid, cudaStream_t s, const CUtensorMap &kmap,
                             const CUtensorMap &qmap, const ImpArgs &a)
{
    switch (pl.stages) {
    case 2:
        return launch(rkv_importance_kernel<NR, 2>, grid, dim3(imp_threads(NR)), ImpSmem<NR, 2>::kAlloc, pl.cluster, s,
                      kmap, qmap, a);
    case 3:
        return launch(rkv_importance_kernel<NR, 3>, grid, dim3(imp_threads(NR)), ImpSmem<NR, 3>::kAlloc, pl.cluster, s,
                      kmap, qmap, a);
    default:
        return launch(rkv_importance_kernel<NR, 4>, grid, dim3(imp_threads(NR)), ImpSmem<NR, 4>::kAlloc, pl.cluster, s,
                      kmap, qmap, a);
    }
}

// Which importance kernel runs: the persistent one (clusters walking the
// heads) or the one-shot one (one cluster per head). 1 (default): persistent
// for 64-row query blocks, one-shot for 32-row ones; 0: always one-shot;
// 2: always persistent. Measured on B300: with 64 query rows per head the
// persistent kernel is 22-33% faster (paged Qwen2-7B cache 2051 -> 1377 us,
// N = 4352 at window 16: 1709 -> 1336 us); with 32 rows the one-shot kernel,
// two CTAs per SM, is 6-8% faster (its second CTA streams while the first
// finishes a head).
#ifndef RKV_IMP_PERSISTENT
#define RKV_IMP_PERSISTENT 1
#endif

// Persistent importance: T tiles per CTA, two TMEM halves (consecutive heads)
// when 2 * T * NR <= 512 columns with a cluster of at most 8, else one half.
// (A cluster of one CTA per head, all of a Llama-8B head's 9 tiles in one
// CTA's TMEM, measured no faster on B300: 28.0 against 28.5 us.)
#ifndef RKV_IMP_PT
#define RKV_IMP_PT 0 // > 0: tiles per CTA of the persistent kernel (cluster = ceil(tiles / RKV_IMP_PT))
#endif
ImpPlan plan_importance_persistent(const Geom &g)
{
    ImpPlan pl;
    pl.nr = g.rows <= 32 ? 32 : 64;
    const int tiles_max = ceil_div(g.nmax, kTileKeys);
    // 64 query rows and at most 10 key tiles (a head too wide for one CTA's
    // TMEM, narrow enough for two): two CTAs of ceil(tiles / 2) tiles, one TMEM
    // buffer. Measured on B300 on the paged Qwen2-7B cache (9 tiles): 1244
    // against 1371 us for three CTAs of three tiles, double-buffered; at 34
    // tiles more CTAs per head lost (seven of five tiles: 1967 against 1418 us).
    const int pt = RKV_IMP_PT > 0 ? RKV_IMP_PT : (pl.nr == 64 && tiles_max <= 10 ? (tiles_max + 1) / 2 : 0);
    if (pt > 0 && ceil_div(tiles_max, pt) <= kMaxCluster) {
        const int c = ceil_div(tiles_max, pt);
        pl.tiles_per_cta = ceil_div(tiles_max, c);
        pl.cluster = ceil_div(tiles_max, pl.tiles_per_cta);
        const bool dbl = 2 * pl.tiles_per_cta * pl.nr <= 512;
        pl.tmem_cols = pow2_at_least(static_cast<uint32_t>((dbl ? 2 : 1) * pl.tiles_per_cta * pl.nr));
        pl.stages = 0;
        return pl;
    }
    int c = ceil_div(tiles_max, std::min(kImpMaxTiles, 256 / pl.nr));
    const bool dbl = c <= kMaxCluster;
    if (!dbl)
        c = ceil_div(tiles_max, std::min(kImpMaxTiles, 512 / pl.nr));
    pl.tiles_per_cta = ceil_div(tiles_max, c);
    pl.cluster = ceil_div(tiles_max, pl.tiles_per_cta);
    pl.tmem_cols = pow2_at_least(static_cast<uint32_t>((dbl ? 2 : 1) * pl.tiles_per_cta * pl.nr));
    pl.stages = 0;
    return pl;
}

template <int NR, bool kClosed = false>
rkv_status launch_importance_persistent(const ImpPlan &pl, long long heads, cudaStream_t s, const CUtensorMap &kmap,
                                        const CUtensorMap &qmap, const ImpArgs &a)
{
    auto kernel = rkv_importance_pkernel<NR, kClosed>;
    const size_t smem = ImpPSmem<NR, kClosed>::kAlloc;
    if (!ensure_smem_limit(reinterpret_cast<const void *>(kernel), smem))
        return RKV_ERR_CUDA;
    // clusters resident at once (cached per device and cluster size)
    static std::atomic<int> cache[kMaxDevices][kMaxCluster + 1];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess)
        return RKV_ERR_CUDA;
    int resident = dev < kMaxDevices ? cache[dev][pl.cluster].load(std::memory_order_relaxed) : 0;
    if (resident == 0) {
        cudaLaunchConfig_t cfg = {};
        const int sms = sm_count();
        cfg.gridDim = dim3(static_cast<unsigned>(std::max(pl.cluster, sms - sms % pl.cluster)));
        cfg.blockDim = dim3(imp_threads(NR));
        cfg.dynamicSmemBytes = smem;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = static_cast<unsigned>(pl.cluster);
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        if (cudaOccupancyMaxActiveClusters(&resident, kernel, &cfg) != cudaSuccess || resident < 1)
            resident = std::max(1, sms / pl.cluster);
        if (dev < kMaxDevices)
            cache[dev][pl.cluster].store(resident, std::memory_order_relaxed);
    }
    const long long clusters = std::min<long long>(heads, resident);
    return launch(kernel, dim3(static_cast<unsigned>(clusters * pl.cluster)), dim3(imp_threads(NR)), smem,
                  pl.cluster, s, kmap, qmap, a);
}

// red != nullptr: also the closed-form redundancy, in the same pass over K
// (the persistent kernel with kClosed, whatever RKV_IMP_PERSISTENT says).
rkv_status run_importance(const Geom &g, const void *k, const void *q, float *imp, float *inv, cudaStream_t s,
                          float *red = nullptr)
{
    if (red || RKV_IMP_PERSISTENT == 2 || (RKV_IMP_PERSISTENT == 1 && g.rows > 32)) {
        const ImpPlan pl = plan_importance_persistent(g);
        if (pl.cluster > kMaxCluster || pl.tmem_cols > 512)
            return RKV_ERR_UNSUPPORTED;
        CUtensorMap kmap, qmap;
        if (!encode_k_map(&kmap, g, k) || !encode_q_map(&qmap, g, q, pl.nr))
            return RKV_ERR_CUDA;
        ImpArgs a;
        a.g = g;
        a.out_imp = imp;
        a.out_inv = inv;
        a.out_red = red;
        a.k = static_cast<const uint8_t *>(k);
        a.tiles_per_cta = pl.tiles_per_cta;
        a.tmem_cols = pl.tmem_cols;
        a.scale_log2 = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(kHeadDim)));
        if (red)
            return pl.nr == 32 ? launch_importance_persistent<32, true>(pl, num_heads(g), s, kmap, qmap, a)
                               : launch_importance_persistent<64, true>(pl, num_heads(g), s, kmap, qmap, a);
        if (pl.nr == 32)
            return launch_importance_persistent<32>(pl, num_heads(g), s, kmap, qmap, a);
        return launch_importance_persistent<64>(pl, num_heads(g), s, kmap, qmap, a);
    }
    const ImpPlan pl = plan_importance(g);
    if (pl.cluster > 8 || pl.tmem_cols > 512)
        return RKV_ERR_UNSUPPORTED;
    CUtensorMap kmap, qmap;
    if (!encode_k_map(&kmap, g, k) || !encode_q_map(&qmap, g, q, pl.nr))
        return RKV_ERR_CUDA;
    ImpArgs a;
    a.g = g;
    a.out_imp = imp;
    a.out_inv = inv;
    a.out_red = nullptr;
    a.k = static_cast<const uint8_t *>(k);
    a.tiles_per_cta = pl.tiles_per_cta;
    a.tmem_cols = pl.tmem_cols;
    a.scale_log2 = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(kHeadDim)));
    const dim3 grid(static_cast<unsigned>(num_heads(g) * pl.cluster));
    if (pl.nr == 32)
        return launch_importance<32>(pl, grid, s, kmap, qmap, a);
    return launch_importance<64>(pl, grid, s, kmap, qmap, a);
}

rkv_status run_redundancy_closed(const Geom &g, const void *k, const float *inv, float *red, cudaStream_t s)
{
    const long long heads = num_heads(g);
    const int sms = sm_count();
    if (sms < 1)
        return RKV_ERR_CUDA;
    // Resident rows (K read once): a cluster of C CTAs per head, each holding
    // about RKV_CF_RES_ROWS rows (~36 KB of shared memory, several CTAs per
    // SM), C <= 8.
#ifndef RKV_CF_RES_ROWS
#define RKV_CF_RES_ROWS 144 // 0: always the streaming kernel
#endif
    // Measured on B300: resident rows win for heads of up to ~1280 keys (a
    // paged Qwen2-7B cache: 2.99 against 3.12 ms for steps 1-2); for longer
    // heads a CTA holds 272+ rows, fewer CTAs fit an SM, and the streaming
    // kernel is faster (N = 4352: 3.27 against 5.28 ms).
#ifndef RKV_CF_RES_MAX_ROWS
#define RKV_CF_RES_MAX_ROWS 160
#endif
    if (RKV_CF_RES_ROWS > 0) {
        const int c = std::min(8, std::max(1, ceil_div(g.nmax, RKV_CF_RES_ROWS)));
        const int rows = ceil_div(ceil_div(g.nmax, c), 16) * 16;
        // Persistent clusters walking the heads, rows brought in by TMA (the
        // next head's during this one's passes).
#ifndef RKV_CF_PERSISTENT
#define RKV_CF_PERSISTENT 1
#endif
        if (RKV_CF_PERSISTENT && rows <= kCfpMaxRows) {
            CUtensorMap kmap;
            if (!encode_k_rows_map(&kmap, g, k, rows))
                return RKV_ERR_CUDA;
            auto kernel = rkv_redundancy_closed_pkernel;
            if (!ensure_smem_limit(reinterpret_cast<const void *>(kernel), CfpSmem::kAlloc))
                return RKV_ERR_CUDA;
            static std::atomic<int> cache[kMaxDevices][9];
            int dev = 0;
            if (cudaGetDevice(&dev) != cudaSuccess)
                return RKV_ERR_CUDA;
            int resident = dev < kMaxDevices ? cache[dev][c].load(std::memory_order_relaxed) : 0;
            if (resident == 0) {
                cudaLaunchConfig_t cfg = {};
                cfg.gridDim = dim3(static_cast<unsigned>(std::max(c, sms - sms % c)));
                cfg.blockDim = dim3(kCfpThreads);
                cfg.dynamicSmemBytes = CfpSmem::kAlloc;
                cudaLaunchAttribute attr[1];
                attr[0].id = cudaLaunchAttributeClusterDimension;
                attr[0].val.clusterDim.x = static_cast<unsigned>(c);
                attr[0].val.clusterDim.y = 1;
                attr[0].val.clusterDim.z = 1;
                cfg.attrs = attr;
                cfg.numAttrs = 1;
                if (cudaOccupancyMaxActiveClusters(&resident, kernel, &cfg) != cudaSuccess || resident < 1)
                    resident = std::max(1, sms / c);
                if (dev < kMaxDevices)
                    cache[dev][c].store(resident, std::memory_order_relaxed);
            }
            CfArgs a;
            a.g = g;
            a.k = static_cast<const uint8_t *>(k);
            a.inv = inv;
            a.out_red = red;
            a.rows_per_cta = rows;
            const long long clusters = std::min<long long>(heads, resident);
            return launch(kernel, dim3(static_cast<unsigned>(clusters * c)), dim3(kCfpThreads),
                             CfpSmem::kAlloc, c, s, kmap, a);
        }
        const size_t smem = cf_res_smem_bytes(rows);
        if (rows <= RKV_CF_RES_MAX_ROWS && smem <= 220u * 1024u) {
            CfArgs a;
            a.g = g;
            a.k = static_cast<const uint8_t *>(k);
            a.inv = inv;
            a.out_red = red;
            a.rows_per_cta = rows;
            return launch(rkv_redundancy_closed_res_kernel, dim3(static_cast<unsigned>(heads * c)),
                          dim3(kCfResThreads), smem, c, s, a);
        }
    }
    // Streaming: a power-of-two cluster up to 8, grown until the grid has
    // about six CTAs per SM, keeping at least 128 rows per CTA.
    int c = 1;
    while (c < 8 && heads * c < 6ll * sms && g.nmax / (2 * c) >= 128)
        c *= 2;
    CfArgs a;
    a.g = g;
    a.k = static_cast<const uint8_t *>(k);
    a.inv = inv;
    a.out_red = red;
    a.rows_per_cta = ceil_div(ceil_div(g.nmax, c), kCfRowsPerPass) * kCfRowsPerPass;
    return launch(rkv_redundancy_closed_kernel, dim3(static_cast<unsigned>(heads * c)),
                     dim3(kCfThreads), 0, c, s,
                  a);
}

// The CTA-pair Gram kernel, persistent: as many CTA pairs as can be resident
// at once (an SM left without a partner in its GPC cannot host one).
rkv_status launch_pair_gram(const CUtensorMap &kmap, const RedArgs &a, long long items, int sms, cudaStream_t s)
{
    static std::atomic<int> max_pairs[kMaxDevices];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess)
        return RKV_ERR_CUDA;
    int resident = dev < kMaxDevices ? max_pairs[dev].load(std::memory_order_relaxed) : 0;
    if (resident == 0) {
        if (!ensure_smem_limit(reinterpret_cast<const void *>(rkv_redundancy_pair_kernel), PairSmem::kAlloc))
            return RKV_ERR_CUDA;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(static_cast<unsigned>(sms & ~1));
        cfg.blockDim = dim3(kPairThreads);
        cfg.dynamicSmemBytes = PairSmem::kAlloc;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 2;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        if (cudaOccupancyMaxActiveClusters(&resident, rkv_redundancy_pair_kernel, &cfg) != cudaSuccess ||
            resident < 1)
            resident = sms / 2;
        if (dev < kMaxDevices)
            max_pairs[dev].store(resident, std::memory_order_relaxed);
    }
    const dim3 grid(static_cast<unsigned>(2 * std::min<long long>(items, resident)));
    return launch(rkv_redundancy_pair_kernel, grid, dim3(kPairThreads), PairSmem::kAlloc, 2, s, kmap,
                     a);
}

rkv_status run_redundancy(const Geom &g, const void *k, const float *inv, float *red, cudaStream_t s)
{
    if (g.redundancy != RKV_REDUNDANCY_GRAM) // either closed form: from the inverse norms given
        return run_redundancy_closed(g, k, inv, red, s);
    CUtensorMap kmap;
    if (!encode_k_map(&kmap, g, k))
        return RKV_ERR_CUDA;
    RedArgs a;
    a.g = g;
    a.inv = inv;
    a.out_red = red;
    a.pairs = ceil_div(ceil_div(g.nmax, kTileKeys), 2); // 256-row blocks per head
    a.heads = static_cast<int>(num_heads(g));
    const long long items = num_heads(g) * a.pairs;
    if (items > 0x7FFFFFFFll)
        return RKV_ERR_UNSUPPORTED;
    a.item0 = 0;
    a.items = static_cast<int>(items);
    a.interleave = 0;
    int sms = 0;
    if ((sms = sm_count()) < 1)
        return RKV_ERR_CUDA;
    // The CTA-pair kernel works on 256-row blocks and 256-key column tiles:
    // faster per flop on long heads (each SM reads only its own operand
    // halves), but a half 256-row block (the last 128-row tile of an odd tile
    // count) would cost it a whole block. So with an even tile count it takes
    // every item; with an odd count of at least kSplitTiles it takes the full
    // blocks and the single-CTA kernel, launched after it on the same stream,
    // the half blocks (red_item_map deals all full blocks before any half
    // block). Measured on B300: at 9 tiles (N = 1152) the split is 3-9%
    // slower than the single-CTA kernel alone (few 256-key column tiles per
    // item to spread the pair's per-item costs over), at 17 tiles (N = 2176)
    // 7% faster.
#ifndef RKV_RED_PAIR
#define RKV_RED_PAIR 3 // 0: single-CTA kernel, 1: CTA pairs, 2: pairs for even tile counts,
                       // 3: as 2, plus the full blocks of odd counts >= kSplitTiles
#endif
#ifndef RKV_RED_SPLIT_TILES
#define RKV_RED_SPLIT_TILES 17
#endif
    constexpr int kSplitTiles = RKV_RED_SPLIT_TILES;
    const int tiles_max = ceil_div(g.nmax, kTileKeys);
    const bool even = tiles_max % 2 == 0;
    const bool use_pair = sms >= 2 && (RKV_RED_PAIR == 1 || (RKV_RED_PAIR >= 2 && even));
    if (use_pair)
        return launch_pair_gram(kmap, a, items, sms, s);
    const bool split = sms >= 2 && RKV_RED_PAIR == 3 && tiles_max >= kSplitTiles;
    if (split) {
        const long long full = num_heads(g) * (tiles_max / 2);
        RedArgs pa = a;
        pa.items = static_cast<int>(full);
        const rkv_status st = launch_pair_gram(kmap, pa, full, sms, s);
        if (st != RKV_OK)
            return st;
        a.item0 = static_cast<int>(full);
    }
    const dim3 grid(static_cast<unsigned>(std::min<long long>(a.items - a.item0, sms)));
    // Item order for the single-CTA kernel alone (no split launch relies on
    // the full-blocks-first order): a head's blocks together once every CTA
    // has many items (see red_item_map).
#ifndef RKV_RED_INTERLEAVE
#define RKV_RED_INTERLEAVE 1 // 0: full blocks first always; 2: interleaved always
#endif
    if (a.item0 == 0 && (RKV_RED_INTERLEAVE == 2 || (RKV_RED_INTERLEAVE == 1 && a.items >= 16ll * sms)))
        a.interleave = 1;
    // The single-CTA Gram with 128x256 MMAs on both layouts. Measured on
    // B300: Llama-3-8B cache (contiguous, N = 1152) 85.6 -> 76.3 us with the
    // wide form; paged Qwen2-7B cache 4.30 -> 4.18 ms once a head's items are
    // dealt together (with all full blocks first the two forms were even).
#ifndef RKV_RED_WIDE
#define RKV_RED_WIDE 2 // 0: never the wide form; 1: on the contiguous layout; 2: on both layouts
#endif
    if (RKV_RED_WIDE == 2 || (RKV_RED_WIDE == 1 && !g.paged))
        return launch(rkv_redundancy_wide_kernel, grid, dim3(kWideThreads), WideSmem::kAlloc, 1, s,
                         kmap, a);
    return launch(rkv_redundancy_kernel, grid, dim3(kRedThreads), RedSmem::kAlloc, 1, s, kmap, a);
}

rkv_status run_select(const Geom &g, const float *imp, const float *red, int32_t *keep, float *scores,
                      cudaStream_t s)
{
    SelArgs a;
    a.g = g;
    a.imp = imp;
    a.red = red;
    a.keep = keep;
    a.scores = scores;
    if (g.shared_sel) {
        const size_t smem = sel_smem_bytes(g.npad, true);
        return launch(rkv_select_kernel<true>, dim3(static_cast<unsigned>(num_heads(g) / g.Hkv)), dim3(kSelThreads),
                      smem, 1, s, a);
    }
    const size_t smem = sel_smem_bytes(g.npad, false);
    return launch(rkv_select_kernel<false>, dim3(static_cast<unsigned>(num_heads(g))), dim3(kSelThreads), smem, 1, s,
                  a);
}

int compact_cluster(const Geom &g, int sms);

rkv_status run_compact(const Geom &g, void *k, void *v, const int32_t *keep, int32_t *freed_off,
                       int32_t *freed_ids, int32_t *new_lens, cudaStream_t s)
{
    CompactArgs a;
    a.g = g;
    a.k = static_cast<uint8_t *>(k);
    a.v = static_cast<uint8_t *>(v);
    a.keep = keep;
    a.freed_off = freed_off;
    a.freed_ids = freed_ids;
    a.new_lens = new_lens;
    const int sms = sm_count();
    if (sms < 1)
        return RKV_ERR_CUDA;
    const int c = compact_cluster(g, sms);
    const dim3 grid(static_cast<unsigned>(num_heads(g) * c));
    return launch(rkv_compact_kernel, grid, dim3(kCpThreads), 0, c, s, a);
}

// Cluster size of the compaction kernels: a power of two up to 8, grown until
// the grid has about six CTAs per SM, and no larger than the budget's 64-row
// rounds.
int compact_cluster(const Geom &g, int sms)
{
#ifndef RKV_CP_TARGET
#define RKV_CP_TARGET 6
#endif
    const long long heads = num_heads(g);
    int c = 1;
    while (c < 8 && heads * c < RKV_CP_TARGET * static_cast<long long>(sms) && 2 * c * kCpRows <= g.budget)
        c *= 2;
    return c;
}

// Steps 3-5 in one launch (per-KV-head selection only). Returns
// RKV_ERR_UNSUPPORTED when the selection scratch does not fit a CTA's shared
// memory, in which case the caller runs rkv_select and rkv_compact instead.
#ifndef RKV_SCP_FUSED
#define RKV_SCP_FUSED 1 // 0: never fuse (rkv_compress runs the separate select and compact kernels)
#endif
rkv_status run_select_compact(const Geom &g, const float *imp, const float *red, void *k, void *v, int32_t *keep,
                              float *scores, int32_t *freed_off, int32_t *freed_ids, int32_t *new_lens,
                              cudaStream_t s)
{
    if (g.shared_sel || !RKV_SCP_FUSED)
        return RKV_ERR_UNSUPPORTED;
    const size_t smem = selcp_smem_bytes(g.npad, g.budget);
    if (smem + sizeof(int32_t) * (kMaxSeq / kBlock) + 64 > 227u * 1024u)
        return RKV_ERR_UNSUPPORTED;
    const int sms = sm_count();
    if (sms < 1)
        return RKV_ERR_CUDA;
    SelCompactArgs a;
    a.c.g = g;
    a.c.k = static_cast<uint8_t *>(k);
    a.c.v = static_cast<uint8_t *>(v);
    a.c.keep = keep;
    a.c.freed_off = freed_off;
    a.c.freed_ids = freed_ids;
    a.c.new_lens = new_lens;
    a.s.g = g;
    a.s.imp = imp;
    a.s.red = red;
    a.s.keep = keep;
    a.s.scores = scores;
    // One 512-thread CTA per head instead of a cluster per head, once there
    // are at least as many heads as SMs: the cluster's peers then no longer
    // idle at the barrier while their rank 0 selects. With fewer heads the
    // cluster spreads the row moves of each head over more SMs.
#ifndef RKV_SCP_SOLO
#define RKV_SCP_SOLO 2 // 0: never, 1: always, 2: when heads >= SMs
#endif
    if (RKV_SCP_SOLO == 1 || (RKV_SCP_SOLO == 2 && num_heads(g) >= sms)) {
        const size_t ssmem = selcp_solo_smem_bytes(g.npad, g.budget);
        if (2 * (ssmem + sizeof(int32_t) * (kMaxSeq / kBlock) + 64) <= 227u * 1024u)
            return launch(rkv_select_compact_solo_kernel, dim3(static_cast<unsigned>(num_heads(g))),
                          dim3(kScpSoloThreads), ssmem, 1, s, a);
    }
    const int c = compact_cluster(g, sms);
    const long long ctas = num_heads(g) * c;
    const dim3 grid(static_cast<unsigned>(ctas));
    return launch(rkv_select_compact_kernel, grid, dim3(kCpThreads), smem, c, s, a);
}

struct Workspace {
    float *imp, *red, *inv;
};

// Steps 1-2: importance, then the redundancy kernel (dense Gram or closed
// form); with RKV_REDUNDANCY_CLOSED_FORM_FUSED one launch of the importance
// kernel that also forms R from the same pass over K (if the persistent
// importance kernel cannot take the problem, the two-kernel closed form).
rkv_status run_importance_redundancy(const Geom &g, const void *k, const void *q, float *imp, float *inv, float *red,
                                     cudaStream_t s)
{
    if (g.redundancy == RKV_REDUNDANCY_CLOSED_FORM_FUSED) {
        const rkv_status st = run_importance(g, k, q, imp, inv, s, red);
        if (st != RKV_ERR_UNSUPPORTED)
            return st;
    }
    const rkv_status st = run_importance(g, k, q, imp, inv, s);
    if (st != RKV_OK)
        return st;
    return run_redundancy(g, k, inv, red, s);
}

size_t workspace_bytes_for(const Geom &g)
{
    const size_t plane = (static_cast<size_t>(num_heads(g)) * g.npad * 4 + 255) & ~size_t(255);
    return 3 * plane;
}

} // namespace

// Marks the launches of one entry-point call as those of a small problem
// (fewer heads than SMs) or not, for RKV_PDL 2.
struct PdlScope {
    bool prev;
    explicit PdlScope(const Geom &g) : prev(t_small_problem)
    {
        t_small_problem = num_heads(g) < static_cast<long long>(sm_count());
    }
    ~PdlScope() { t_small_problem = prev; }
    PdlScope(const PdlScope &) = delete;
    PdlScope &operator=(const PdlScope &) = delete;
};

extern "C" {

const char *rkv_status_string(rkv_status status)
{
    switch (status) {
    case RKV_OK: return "ok";
    case RKV_ERR_INVALID_ARG: return "invalid argument";
    case RKV_ERR_WORKSPACE: return "workspace missing or too small";
    case RKV_ERR_UNSUPPORTED: return "unsupported problem";
    case RKV_ERR_CUDA: return "CUDA error";
    case RKV_ERR_DEVICE: return "invalid device-side input (seq_lens, block table or kept indices)";
    case RKV_ERR_TIMEOUT: return "bounded in-kernel wait timed out";
    }
    return "unknown status";
}

int rkv_version(void) { return 600; }

int32_t rkv_score_stride(const rkv_problem *p)
{
    if (!p || p->max_seq_len < 1)
        return 0;
    return ceil_div(p->max_seq_len, kTileKeys) * kTileKeys;
}

rkv_status rkv_workspace_size(const rkv_problem *p, size_t *bytes)
{
    if (!bytes)
        return RKV_ERR_INVALID_ARG;
    const rkv_status st = check_problem(p);
    if (st != RKV_OK)
        return st;
    *bytes = workspace_bytes_for(make_geom(p, nullptr, nullptr));
    return RKV_OK;
}

rkv_status rkv_importance(const rkv_problem *p, const void *k_cache, const void *q_window, const int32_t *seq_lens,
                          const int32_t *block_table, float *out_importance, float *out_inv_norm,
                          cudaStream_t stream)
{
    rkv_status st = check_problem(p);
    if (st != RKV_OK)
        return st;
    if (!k_cache || !q_window || !seq_lens || !out_importance || !out_inv_norm ||
        (p->layout == RKV_LAYOUT_PAGED && !block_table))
        return RKV_ERR_INVALID_ARG;
    if (!aligned16(k_cache) || !aligned16(q_window) || !aligned16(out_importance) || !aligned16(out_inv_norm))
        return RKV_ERR_INVALID_ARG;
    const Geom g = make_geom(p, seq_lens, block_table);
    const PdlScope pdl_scope(g);
    if (num_heads(g) == 0)
        return RKV_OK;
    return run_importance(g, k_cache, q_window, out_importance, out_inv_norm, stream);
}

rkv_status rkv_importance_redundancy(const rkv_problem *p, const void *k_cache, const void *q_window,
                                     const int32_t *seq_lens, const int32_t *block_table, float *out_importance,
                                     float *out_inv_norm, float *out_redundancy, cudaStream_t stream)
{
    rkv_status st = check_problem(p);
    if (st != RKV_OK)
        return st;
    if (!k_cache || !q_window || !seq_lens || !out_importance || !out_inv_norm || !out_redundancy ||
        (p->layout == RKV_LAYOUT_PAGED && !block_table))
        return RKV_ERR_INVALID_ARG;
    if (!aligned16(k_cache) || !aligned16(q_window) || !aligned16(out_importance) || !aligned16(out_inv_norm) ||
        !aligned16(out_redundancy))
        return RKV_ERR_INVALID_ARG;
    const Geom g = make_geom(p, seq_lens, block_table);
    const PdlScope pdl_scope(g);
    if (num_heads(g) == 0)
        return RKV_OK;
    return run_importance_redundancy(g, k_cache, q_window, out_importance, out_inv_norm, out_redundancy, stream);
}

rkv_status rkv_redundancy(const rkv_problem *p, const void *k_cache, const int32_t *seq_lens,
                          const int32_t *block_table, const float *inv_norm, float *out_redundancy,
                          cudaStream_t stream)
{
    rkv_status st = check_problem(p);
    if (st != RKV_OK)
        return st;
    if (!k_cache || !seq_lens || !inv_norm || !out_redundancy || (p->layout == RKV_LAYOUT_PAGED && !block_table))
        return RKV_ERR_INVALID_ARG;
    if (!aligned16(k_cache) || !aligned16(inv_norm) || !aligned16(out_redundancy))
        return RKV_ERR_INVALID_ARG;
    const Geom g = make_geom(p, seq_lens, block_table);
    const PdlScope pdl_scope(g);
    if (num_heads(g) == 0)
        return RKV_OK;
    return run_redundancy(g, k_cache, inv_norm, out_redundancy, stream);
}

rkv_status rkv_select(const rkv_problem *p, const float *importance, const float *redundancy,
                      const int32_t *seq_lens, int32_t *out_keep_idx, float *out_scores, cudaStream_t stream)
{
    rkv_status st = check_problem(p);
    if (st != RKV_OK)
        return st;
    if (!importance || !redundancy || !seq_lens || !out_keep_idx)
        return RKV_ERR_INVALID_ARG;
    if (!aligned16(importance) || !aligned16(redundancy))
        return RKV_ERR_INVALID_ARG;
    const Geom g = make_geom(p, seq_lens, nullptr);
    const PdlScope pdl_scope(g);
    if (num_heads(g) == 0)
        return RKV_OK;
    return run_select(g, importance, redundancy, out_keep_idx, out_scores, stream);
}

rkv_status rkv_compact(const rkv_problem *p, void *k_cache, void *v_cache, const int32_t *seq_lens,
                       const int32_t *block_table, const int32_t *keep_idx, int32_t *out_freed_off,
                       int32_t *out_freed_ids, int32_t *out_new_seq_lens, cudaStream_t stream)
{
    rkv_status st = check_problem(p);
    if (st != RKV_OK)
        return st;
    const bool paged = p->layout == RKV_LAYOUT_PAGED;
    if (!k_cache || !v_cache || !seq_lens || !keep_idx || !out_freed_off || !out_new_seq_lens ||
        (paged && (!block_table || !out_freed_ids)))
        return RKV_ERR_INVALID_ARG;
    if (!aligned16(k_cache) || !aligned16(v_cache))
        return RKV_ERR_INVALID_ARG;
    const Geom g = make_geom(p, seq_lens, block_table);
    const PdlScope pdl_scope(g);
    if (num_heads(g) == 0) {
        if (g.B == 0)
            return cudaMemsetAsync(out_freed_off, 0, sizeof(int32_t), stream) == cudaSuccess ? RKV_OK
                                                                                                 : RKV_ERR_CUDA;
        return RKV_OK;
    }
    return run_compact(g, k_cache, v_cache, keep_idx, out_freed_off, out_freed_ids, out_new_seq_lens, stream);
}

rkv_status rkv_compress(const rkv_problem *p, void *k_cache, void *v_cache, const void *q_window,
                        const int32_t *seq_lens, const int32_t *block_table, int32_t *out_keep_idx,
                        int32_t *out_freed_off, int32_t *out_freed_ids, int32_t *out_new_seq_lens, float *out_scores,
                        void *workspace, size_t workspace_bytes, cudaStream_t stream)
{
    rkv_status st = check_problem(p);
    if (st != RKV_OK)
        return st;
    const bool paged = p->layout == RKV_LAYOUT_PAGED;
    if (!k_cache || !v_cache || !q_window || !seq_lens || !out_keep_idx || !out_freed_off || !out_new_seq_lens ||
        (paged && (!block_table || !out_freed_ids)))
        return RKV_ERR_INVALID_ARG;
    if (!aligned16(k_cache) || !aligned16(v_cache) || !aligned16(q_window))
        return RKV_ERR_INVALID_ARG;
    const Geom g = make_geom(p, seq_lens, block_table);
    const PdlScope pdl_scope(g);
    if (num_heads(g) == 0)
        return rkv_compact(p, k_cache, v_cache, seq_lens, block_table, out_keep_idx, out_freed_off, out_freed_ids,
                           out_new_seq_lens, stream);
    const size_t need = workspace_bytes_for(g);
    if (!workspace || workspace_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 255u))
        return RKV_ERR_WORKSPACE;
    const size_t plane = need / 3;
    Workspace ws;
    ws.imp = static_cast<float *>(workspace);
    ws.red = reinterpret_cast<float *>(static_cast<uint8_t *>(workspace) + plane);
    ws.inv = reinterpret_cast<float *>(static_cast<uint8_t *>(workspace) + 2 * plane);
    if ((st = run_importance_redundancy(g, k_cache, q_window, ws.imp, ws.inv, ws.red, stream)) != RKV_OK)
        return st;
    st = run_select_compact(g, ws.imp, ws.red, k_cache, v_cache, out_keep_idx, out_scores, out_freed_off,
                            out_freed_ids, out_new_seq_lens, stream);
    if (st != RKV_ERR_UNSUPPORTED)
        return st;
    if ((st = run_select(g, ws.imp, ws.red, out_keep_idx, out_scores, stream)) != RKV_OK)
        return st;
    return run_compact(g, k_cache, v_cache, out_keep_idx, out_freed_off, out_freed_ids, out_new_seq_lens, stream);
}

rkv_status rkv_select_compact(const rkv_problem *p, const float *importance, const float *redundancy,
                              const int32_t *seq_lens, const int32_t *block_table, void *k_cache, void *v_cache,
                              int32_t *out_keep_idx, int32_t *out_freed_off, int32_t *out_freed_ids,
                              int32_t *out_new_seq_lens, float *out_scores, cudaStream_t stream)
{
    rkv_status st = check_problem(p);
    if (st != RKV_OK)
        return st;
    const bool paged = p->layout == RKV_LAYOUT_PAGED;
    if (!importance || !redundancy || !seq_lens || !k_cache || !v_cache || !out_keep_idx || !out_freed_off ||
        !out_new_seq_lens || (paged && (!block_table || !out_freed_ids)))
        return RKV_ERR_INVALID_ARG;
    if (!aligned16(importance) || !aligned16(redundancy) || !aligned16(k_cache) || !aligned16(v_cache))
        return RKV_ERR_INVALID_ARG;
    const Geom g = make_geom(p, seq_lens, block_table);
    const PdlScope pdl_scope(g);
    if (num_heads(g) == 0)
        return rkv_compact(p, k_cache, v_cache, seq_lens, block_table, out_keep_idx, out_freed_off, out_freed_ids,
                           out_new_seq_lens, stream);
    st = run_select_compact(g, importance, redundancy, k_cache, v_cache, out_keep_idx, out_scores, out_freed_off,
                            out_freed_ids, out_new_seq_lens, stream);
    if (st != RKV_ERR_UNSUPPORTED)
        return st;
    if ((st = run_select(g, importance, redundancy, out_keep_idx, out_scores, stream)) != RKV_OK)
        return st;
    return run_compact(g, k_cache, v_cache, out_keep_idx, out_freed_off, out_freed_ids, out_new_seq_lens, stream);
}

rkv_status rkv_free_blocks_push(const int32_t *freed_off, const int32_t *freed_ids, int32_t batch,
                                int32_t *free_stack, int32_t *free_top, int32_t capacity, cudaStream_t stream)
{
    if (batch < 0 || capacity < 0 || !freed_off || !free_top || (capacity > 0 && !free_stack))
        return RKV_ERR_INVALID_ARG;
    return launch(rkv::rkv_free_push_kernel, dim3(1), dim3(kPushThreads), 0, 1, stream, freed_off, freed_ids,
                  static_cast<int>(batch), free_stack, free_top, static_cast<int>(capacity));
}

rkv_status rkv_device_status(cudaStream_t stream)
{
    if (cudaStreamSynchronize(stream) != cudaSuccess)
        return RKV_ERR_CUDA;
    int v = 0;
    if (cudaMemcpyFromSymbol(&v, rkv::g_error, sizeof(int)) != cudaSuccess)
        return RKV_ERR_CUDA;
    if (v != 0) {
        const int zero = 0;
        if (cudaMemcpyToSymbol(rkv::g_error, &zero, sizeof(int)) != cudaSuccess)
            return RKV_ERR_CUDA;
    }
    if (v == kErrDevice)
        return RKV_ERR_DEVICE;
    if (v == kErrTimeout)
        return RKV_ERR_TIMEOUT;
    return RKV_OK;
}

} // extern "C"

// ---------------------------------------------------------------------------
// rkv_compress_noalloc: the same compression event as rkv_compress, for
// callers that cannot hand the library a device workspace. Its scratch (the
// importance, redundancy and inverse-norm planes) lives in the fixed array
// below, which every GPU that loads this library holds until the process
// exits.
static __device__ __align__(256) uint8_t rkv_noalloc_scratch[RKV_NOALLOC_SCRATCH_BYTES];

namespace {

std::mutex g_noalloc_mutex;
struct NoallocEntry {
    unsigned long long ctx_id; // the CUDA context the address belongs to (0: none yet)
    void *ptr;
};
NoallocEntry g_noalloc[kMaxDevices] = {};

// Unique id of the calling thread's current CUDA context (cuCtxGetId), or 0.
unsigned long long current_context_id()
{
    static const auto get_current =
        reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(driver_entry("cuCtxGetCurrent", 4000));
    static const auto get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(driver_entry("cuCtxGetId", 12000));
    if (!get_current || !get_id)
        return 0;
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (get_current(&ctx) != CUDA_SUCCESS || !ctx || get_id(ctx, &id) != CUDA_SUCCESS)
        return 0;
    return id;
}

// Device address of the static scratch in the current device's context. The
// host-side name of the array is only a stand-in; the real address is looked
// up with the device current and cached together with the id of the context
// it belongs to. A context that is torn down and created again (for instance
// after cudaDeviceReset) loads the module again, possibly at another address:
// its new id no longer matches and the address is looked up afresh.
rkv_status noalloc_scratch(void **out)
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return RKV_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_noalloc_mutex);
    NoallocEntry &ent = g_noalloc[dev];
    const unsigned long long ctx = current_context_id(); // 0 before the runtime has made a context
    if (!ent.ptr || ctx == 0 || ent.ctx_id != ctx) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, rkv_noalloc_scratch) != cudaSuccess || !p)
            return RKV_ERR_CUDA;
        ent.ptr = p;
        ent.ctx_id = current_context_id(); // the lookup has made the context current if it was not
    }
    *out = ent.ptr;
    return RKV_OK;
}

} // namespace

extern "C" rkv_status rkv_compress_noalloc(const rkv_problem *p, void *k_cache, void *v_cache,
                                           const void *q_window, const int32_t *seq_lens,
                                           const int32_t *block_table, int32_t *out_keep_idx,
                                           int32_t *out_freed_off, int32_t *out_freed_ids,
                                           int32_t *out_new_seq_lens, float *out_scores, cudaStream_t stream)
{
    rkv_status st = check_problem(p);
    if (st != RKV_OK)
        return st;
    const Geom g = make_geom(p, seq_lens, block_table);
    const PdlScope pdl_scope(g);
    if (num_heads(g) > 0 && workspace_bytes_for(g) > static_cast<size_t>(RKV_NOALLOC_SCRATCH_BYTES))
        return RKV_ERR_WORKSPACE; // the problem needs more scratch than the static array holds
    void *scratch = nullptr;
    if ((st = noalloc_scratch(&scratch)) != RKV_OK)
        return st;
    return rkv_compress(p, k_cache, v_cache, q_window, seq_lens, block_table, out_keep_idx, out_freed_off,
                        out_freed_ids, out_new_seq_lens, out_scores, scratch, RKV_NOALLOC_SCRATCH_BYTES, stream);
}
