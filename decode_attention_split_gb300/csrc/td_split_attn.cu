// Instantiations, launch planning and per-device attribute cache for the split-attention kernel.
#include <algorithm>
#include <mutex>

#include "td_internal.h"
#include "td_split_attn.cuh"
#include "td_split_cluster.cuh"
#include "td_split_mma.cuh"
#include "td_split_q8.cuh"

namespace td {

namespace {

constexpr int kMaxDevices = 64;
constexpr int kKernelSlots = 2 * 2 * 4 + 2 * 2 + 2;  // CUDA-core: dtype x D x row padding; mma: D x m tiles; q8: D

struct KernelRef {
  const void *fn;
  int smem;
  cudaError_t (*launch)(const SplitParams &, int grid, int smem, cudaStream_t);
};

template <typename E, int D, int RP>
cudaError_t launch_one(const SplitParams &p, int grid, int smem, cudaStream_t stream) {
  return launch_pdl(split_attn_kernel<E, D, RP>, dim3(grid), dim3(kThreads), smem, stream, p);
}

template <typename E, int D, int RP>
KernelRef ref_of() {
  if constexpr (SplitCfg<E, D, RP>::kFits) {
    return KernelRef{reinterpret_cast<const void *>(&split_attn_kernel<E, D, RP>), SplitCfg<E, D, RP>::SMEM_BYTES,
                     &launch_one<E, D, RP>};
  } else {
    return KernelRef{nullptr, 0, nullptr};
  }
}

int rp_index(int RP) { return RP == 1 ? 0 : RP == 2 ? 1 : RP == 4 ? 2 : 3; }

// Returns the kernel for (dtype, D, RP); fn == nullptr when not built.
template <typename E>
KernelRef pick_d(int D, int RP) {
  if (D == 64) {
    switch (RP) {
      case 1: return ref_of<E, 64, 1>();
      case 2: return ref_of<E, 64, 2>();
      case 4: return ref_of<E, 64, 4>();
      case 8: return ref_of<E, 64, 8>();
    }
  } else if (D == 128) {
    switch (RP) {
      case 1: return ref_of<E, 128, 1>();
      case 2: return ref_of<E, 128, 2>();
      case 4: return ref_of<E, 128, 4>();
    }
  }
  return KernelRef{nullptr, 0, nullptr};
}

// cuTensorMapEncodeTiled, resolved once through the runtime (no link against the driver).
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}

// 3-D map over a bf16 cache [B*Hkv][Smax][D]: boxes of 64 columns (128 bytes) x 64 rows,
// 128-byte swizzle, zero fill outside the tensor.
bool encode_cache_map(CUtensorMap *map, const void *base, int B, int Hkv, int Smax, int D) {
  const PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (enc == nullptr) return false;
  const cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)Smax, (cuuint64_t)B * Hkv};
  const cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)Smax * D * 2};
  const cuuint32_t box[3] = {64, 64, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The persistent kernel's instantiation for this launch: the tile by the rows; the plan made
// before the wait for the previous kernel when one row block of at most 16 rows covers a kv
// head (decode with grouped heads), after it otherwise (the 24-row tile has no registers to
// spare for the early plan: it spilled).
template <int D>
cudaError_t launch_mma_tile(const MmaArgs &a, int grid, int smem, cudaStream_t stream) {
  const int tile = tile_of_rows(a.p.R);
  if (a.p.RB == 1 && tile == kTileN8)
    return launch_pdl(split_attn_mma_kernel<D, true, kTileN8>, dim3(grid), dim3(kThreads), smem, stream, a);
  if (a.p.RB == 1 && tile == kTileM16)
    return launch_pdl(split_attn_mma_kernel<D, true, kTileM16>, dim3(grid), dim3(kThreads), smem, stream, a);
  if (tile == kTileN8)
    return launch_pdl(split_attn_mma_kernel<D, false, kTileN8>, dim3(grid), dim3(kThreads), smem, stream, a);
  if (tile == kTileM16)
    return launch_pdl(split_attn_mma_kernel<D, false, kTileM16>, dim3(grid), dim3(kThreads), smem, stream, a);
  return launch_pdl(split_attn_mma_kernel<D, false, kTileN24>, dim3(grid), dim3(kThreads), smem, stream, a);
}

template <int D>
cudaError_t launch_mma(const SplitParams &p, int grid, int smem, cudaStream_t stream) {
  MmaArgs a;
  if (!encode_cache_map(&a.kmap, p.k, p.B, p.Hkv, p.Smax, D) || !encode_cache_map(&a.vmap, p.v, p.B, p.Hkv, p.Smax, D))
    return cudaErrorInvalidValue;
  a.p = p;
  {
    // every instantiation's shared-memory opt-in, once per device (the plan's occupancy query
    // set the m16 late-plan one's)
    static std::mutex mu;
    static bool done[kMaxDevices] = {};
    int device = 0;
    if (cudaGetDevice(&device) != cudaSuccess || device < 0 || device >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(mu);
    if (!done[device]) {
      for (const void *fn : {reinterpret_cast<const void *>(&split_attn_mma_kernel<D, true, kTileN8>),
                             reinterpret_cast<const void *>(&split_attn_mma_kernel<D, true, kTileM16>),
                             reinterpret_cast<const void *>(&split_attn_mma_kernel<D, false, kTileN8>),
                             reinterpret_cast<const void *>(&split_attn_mma_kernel<D, false, kTileM16>),
                             reinterpret_cast<const void *>(&split_attn_mma_kernel<D, false, kTileN24>)}) {
        const cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
      }
      done[device] = true;
    }
  }
  return launch_mma_tile<D>(a, grid, smem, stream);
}

template <int D>
KernelRef mma_ref_of() {
  // the ring plus 1024 bytes of slack for its alignment
  constexpr int smem = MmaCfg<D, kPersistentStages<D>>::RING_BYTES + 1024;
  static_assert(smem + 8448 <= 227 * 1024, "mma kernel shared memory");
  return KernelRef{reinterpret_cast<const void *>(&split_attn_mma_kernel<D, false, kTileM16>), smem, &launch_mma<D>};
}

KernelRef pick_mma(int D, int MT) {
  if (MT != 1) return KernelRef{nullptr, 0, nullptr};
  if (D == 64) return mma_ref_of<64>();
  if (D == 128) return mma_ref_of<128>();
  return KernelRef{nullptr, 0, nullptr};
}

// 8-bit caches: 3-D maps over the codes [B*Hkv][Smax][D] (boxes of 128 whole rows, swizzled
// over 128-byte rows for D = 128 and 64-byte rows for D = 64) and 2-D maps over the scales
// [B*Hkv][Smax] (boxes of 132), zero fill outside.
bool encode_q8_maps(Q8Args *a, const SplitParams &p, int D) {
  const PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (enc == nullptr) return false;
  const cuuint32_t estr[3] = {1, 1, 1};
  const cuuint64_t cdims[3] = {(cuuint64_t)D, (cuuint64_t)p.Smax, (cuuint64_t)p.B * p.Hkv};
  const cuuint64_t cstrides[2] = {(cuuint64_t)D, (cuuint64_t)p.Smax * D};
  const cuuint32_t cbox[3] = {(cuuint32_t)D, (cuuint32_t)Q8Cfg<128, kQ8Stages<128>>::TK, 1};
  const cuuint64_t sdims[2] = {(cuuint64_t)p.Smax, (cuuint64_t)p.B * p.Hkv};
  const cuuint64_t sstrides[1] = {(cuuint64_t)p.Smax * 4};
  const cuuint32_t sbox[2] = {Q8Cfg<128, kQ8Stages<128>>::SCALE_BOX, 1};  // a stage's rows plus the alignment slack
  const auto code_map = [&](CUtensorMap *m, const void *base) {
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void *>(base), cdims, cstrides, cbox, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, D == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
  };
  const auto scale_map = [&](CUtensorMap *m, const float *base) {
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float *>(base), sdims, sstrides, sbox, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
  };
  return code_map(&a->kmap, p.k) && code_map(&a->vmap, p.v) && scale_map(&a->ksmap, p.k_scales) &&
         scale_map(&a->vsmap, p.v_scales);
}

template <int D>
cudaError_t launch_q8(const SplitParams &p, int grid, int smem, bool early, cudaStream_t stream) {
  Q8Args a;
  if (!encode_q8_maps(&a, p, D)) return cudaErrorInvalidValue;
  a.p = p;
  if (p.R <= 8) {
    // the narrow instantiations' shared-memory opt-in, once per device (the plan's occupancy
    // query set the other's)
    static std::mutex mu;
    static bool done[kMaxDevices] = {};
    int device = 0;
    if (cudaGetDevice(&device) != cudaSuccess || device < 0 || device >= kMaxDevices) return cudaErrorInvalidDevice;
    {
      std::lock_guard<std::mutex> lock(mu);
      if (!done[device]) {
        for (const void *fn : {reinterpret_cast<const void *>(&split_attn_q8_kernel<D, true, false>),
                               reinterpret_cast<const void *>(&split_attn_q8_kernel<D, true, true>)}) {
          const cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
          if (e != cudaSuccess) return e;
        }
        done[device] = true;
      }
    }
    if (early) return launch_pdl(split_attn_q8_kernel<D, true, true>, dim3(grid), dim3(kThreads), smem, stream, a);
    return launch_pdl(split_attn_q8_kernel<D, true, false>, dim3(grid), dim3(kThreads), smem, stream, a);
  }
  return launch_pdl(split_attn_q8_kernel<D, false, false>, dim3(grid), dim3(kThreads), smem, stream, a);
}

template <int D>
KernelRef q8_ref_of() {
  constexpr int smem = Q8Cfg<D, kQ8Stages<D>>::SMEM_BYTES;
  static_assert(smem + 8704 <= 227 * 1024, "q8 kernel shared memory");
  return KernelRef{reinterpret_cast<const void *>(&split_attn_q8_kernel<D, false, false>), smem, nullptr};
}

template <int D>
constexpr int cluster_smem() {
  return MmaCfg<D, kClusterStages<D>>::RING_BYTES + 1024;  // the ring plus alignment slack
}
static_assert(cluster_smem<128>() + 1024 <= 227 * 1024 && cluster_smem<64>() + 1024 <= 227 * 1024,
              "cluster kernel shared memory");

const void *cluster_fn(int D, int tile) {
  if (D == 64) {
    if (tile == kTileN8) return reinterpret_cast<const void *>(&split_attn_cluster_kernel<64, kTileN8>);
    if (tile == kTileM16) return reinterpret_cast<const void *>(&split_attn_cluster_kernel<64, kTileM16>);
    return reinterpret_cast<const void *>(&split_attn_cluster_kernel<64, kTileN24>);
  }
  if (tile == kTileN8) return reinterpret_cast<const void *>(&split_attn_cluster_kernel<128, kTileN8>);
  if (tile == kTileM16) return reinterpret_cast<const void *>(&split_attn_cluster_kernel<128, kTileM16>);
  return reinterpret_cast<const void *>(&split_attn_cluster_kernel<128, kTileN24>);
}

cudaLaunchConfig_t cluster_config(int D, int grid, int cs, cudaStream_t stream, cudaLaunchAttribute *attr) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = D == 64 ? cluster_smem<64>() : cluster_smem<128>();
  cfg.stream = stream;
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = cs;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cfg;
}

template <int D>
cudaError_t launch_cluster(const SplitParams &p, int grid, int cs, cudaStream_t stream) {
  MmaArgs a;
  if (!encode_cache_map(&a.kmap, p.k, p.B, p.Hkv, p.Smax, D) || !encode_cache_map(&a.vmap, p.v, p.B, p.Hkv, p.Smax, D))
    return cudaErrorInvalidValue;
  a.p = p;
  cudaLaunchAttribute attr[2];
  const cudaLaunchConfig_t cfg = cluster_config(D, grid, cs, stream, attr);
  switch (tile_of_rows(p.R)) {
    case kTileN8: return cudaLaunchKernelEx(&cfg, split_attn_cluster_kernel<D, kTileN8>, a);
    case kTileM16: return cudaLaunchKernelEx(&cfg, split_attn_cluster_kernel<D, kTileM16>, a);
    default: return cudaLaunchKernelEx(&cfg, split_attn_cluster_kernel<D, kTileN24>, a);
  }
}

// variant: row padding RP of the CUDA-core kernel, or m tiles MT of the tensor-core kernel
KernelRef pick(td_dtype dtype, int D, bool mma, int variant) {
  if (mma) return pick_mma(D, variant);
  return dtype == TD_F32 ? pick_d<float>(D, variant) : pick_d<__nv_bfloat16>(D, variant);
}

int slot_of(td_dtype dtype, int D, bool mma, int variant) {
  if (mma) return 16 + (D == 64 ? 0 : 2) + (variant == 1 ? 0 : 1);
  return ((dtype == TD_F32 ? 0 : 1) * 2 + (D == 64 ? 0 : 1)) * 4 + rp_index(variant);
}

std::mutex g_mu;
int g_sms[kMaxDevices];
int g_l2[kMaxDevices];  // L2 bytes (0 = not yet queried)
int g_blocks[kMaxDevices][kKernelSlots];  // resident CTAs per SM (0 = not yet queried)
int g_clusters[kMaxDevices][2][4];         // co-resident clusters of 2, 4, 8, 16 CTAs (+1; 0 = not yet queried)

// Sets the shared-memory opt-in once per device and returns the resident CTAs per SM.
int blocks_per_sm(int device, int slot, const KernelRef &k) {
  std::lock_guard<std::mutex> lock(g_mu);
  if (device >= 0 && device < kMaxDevices && g_blocks[device][slot] > 0) return g_blocks[device][slot];
  if (cudaFuncSetAttribute(k.fn, cudaFuncAttributeMaxDynamicSharedMemorySize, k.smem) != cudaSuccess) return 0;
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k.fn, kThreads, k.smem) != cudaSuccess) return 0;
  if (device >= 0 && device < kMaxDevices) g_blocks[device][slot] = n;
  return n;
}

// Clusters of `cs` CTAs (2, 4, 8 or 16) of the cluster kernel that the device holds at once;
// sets the shared-memory and cluster-size opt-ins of every instantiation on first use and
// asks about the one with the most registers (the 24-row narrow tile's). 0 on error.
int active_clusters(int device, int D, int cs) {
  const int di = D == 64 ? 0 : 1, ci = cs == 2 ? 0 : cs == 4 ? 1 : cs == 8 ? 2 : 3;
  std::lock_guard<std::mutex> lock(g_mu);
  if (device < 0 || device >= kMaxDevices) return 0;
  if (g_clusters[device][di][ci] > 0) return g_clusters[device][di][ci] - 1;
  cudaLaunchAttribute attr[2];
  cudaLaunchConfig_t cfg = cluster_config(D, cs, cs, nullptr, attr);
  cfg.numAttrs = 1;  // the cluster shape alone
  int n = 0;
  bool ok = true;
  for (const int tile : {kTileN8, kTileM16, kTileN24}) {
    const void *fn = cluster_fn(D, tile);
    ok = ok &&
         cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)cfg.dynamicSmemBytes) ==
             cudaSuccess &&
         cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) == cudaSuccess;
  }
  if (!ok || cudaOccupancyMaxActiveClusters(&n, cluster_fn(D, kTileN24), &cfg) != cudaSuccess) {
    cudaGetLastError();
    n = 0;
  }
  g_clusters[device][di][ci] = n + 1;
  return n;
}

size_t align256(size_t x) { return (x + 255) / 256 * 256; }

}  // namespace

int device_sm_count(int device) {
  {
    std::lock_guard<std::mutex> lock(g_mu);
    if (device >= 0 && device < kMaxDevices && g_sms[device] > 0) return g_sms[device];
  }
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, device) != cudaSuccess) return 0;
  std::lock_guard<std::mutex> lock(g_mu);
  if (device >= 0 && device < kMaxDevices) g_sms[device] = n;
  return n;
}

static int device_l2_bytes(int device) {
  {
    std::lock_guard<std::mutex> lock(g_mu);
    if (device >= 0 && device < kMaxDevices && g_l2[device] > 0) return g_l2[device];
  }
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrL2CacheSize, device) != cudaSuccess) return 0;
  std::lock_guard<std::mutex> lock(g_mu);
  if (device >= 0 && device < kMaxDevices) g_l2[device] = n;
  return n;
}

td_status plan_split(td_dtype dtype, int B, int Hq, int Hkv, int T, int Smax, int D, int split, SplitPlan *plan,
                     bool q8) {
  if (dtype != TD_F32 && dtype != TD_BF16) return TD_ERR_UNSUPPORTED;
  if (D != 64 && D != 128) return TD_ERR_UNSUPPORTED;
  if (B < 1 || Hq < 1 || Hkv < 1 || T < 1 || Smax < 1 || split < 0 || Hq % Hkv != 0) return TD_ERR_INVALID_ARG;
  if (B > TD_MAX_BATCH || Smax > (1 << 30) || T > Smax) return TD_ERR_UNSUPPORTED;
  const long long GT = (long long)(Hq / Hkv) * T;
  // bf16 caches: tensor-core kernels, the group's rows split evenly over row blocks of at most
  // 24 rows (tile_of_rows: up to 8 on the narrow n8 tile, 9 to 16 on one m16 tile, 17 to 24 on
  // three n8 tiles, so a 24-row verify chunk reads each K/V tile once); the 8-bit cache kernel
  // has no 24-row tile and takes blocks of at most 16 rows. fp32 caches: CUDA-core kernel, up
  // to 4 (D = 128) or 8 (D = 64) rows per CTA
  const bool mma = dtype == TD_BF16;
  int R, variant;
  if (mma) {
    variant = 1;
    const long long most = q8 ? 16 : kMaxTileRows;
    const long long blocks = (GT + most - 1) / most;
    R = (int)((GT + blocks - 1) / blocks);
  } else {
    const int rmax = D == 128 ? 4 : 8;
    R = (int)(GT < rmax ? GT : rmax);
    variant = 1;
    while (variant < R) variant <<= 1;
    // a 512-byte fp32 row makes a one-row CTA's 32-key stages too large: pad to two rows
    if (dtype == TD_F32 && D == 128 && variant < 2) variant = 2;
  }
  const long long RB = (GT + R - 1) / R;
  const long long U = (long long)Hkv * RB;
  if (q8 && !mma) return TD_ERR_UNSUPPORTED;
  const KernelRef k = q8 ? (D == 64 ? q8_ref_of<64>() : q8_ref_of<128>()) : pick(dtype, D, mma, variant);
  if (k.fn == nullptr) return TD_ERR_UNSUPPORTED;
  int device = 0;
  if (cudaGetDevice(&device) != cudaSuccess) return TD_ERR_CUDA;
  const int sms = device_sm_count(device);
  const int per_sm = blocks_per_sm(device, q8 ? 20 + (D == 64 ? 0 : 1) : slot_of(dtype, D, mma, variant), k);
  if (sms <= 0 || per_sm <= 0) return TD_ERR_CUDA;
  // CTAs the automatic split aims to fill. When a kv head's rows fit one row block and the
  // groups are few, leave one slot per group free: the previous call's merging CTAs (one per
  // group) hold theirs until it ends, and with the slots to spare every CTA of this call is
  // resident early enough to warm L2 with its first stages before that end (3B-style layer,
  // B = 1: 32k 26.3 -> 25.7 us, 16k 17.75 -> 17.4 us; the 8-bit cache with its early plan,
  // see split_attn_q8_kernel; the two-row-block verify is slower this way, 27.5 -> 28.3 us,
  // and keeps the full grid). Only while the groups are at most 1/16 of the slots: 64 groups
  // of the 8-bit kernel (B = 8) lost 13-15 % this way.
  const long long slots = (long long)sms * per_sm;
  const bool spare = mma && RB == 1 && (long long)B * U * 16 <= slots;
  const long long p_target = slots - (spare ? (long long)B * U : 0);
  long long ns;
  if (split > 0) {
    ns = ((long long)Smax + split - 1) / split;
  } else {
    const long long by_size = ((long long)Smax + 15) / 16;
    const long long by_grid = (p_target + U - 1) / U;
    ns = by_size < by_grid ? by_size : by_grid;
    if (ns < 1) ns = 1;
  }
  const long long items_max = (long long)B * U * ns;
  if (items_max >= (1LL << 31)) return TD_ERR_UNSUPPORTED;
  plan->mma = mma;
  plan->q8 = q8;
  plan->RP = variant;
  plan->R = R;
  plan->RB = (int)RB;
  plan->ns_ws = (int)ns;
  plan->p_target = (int)p_target;
  plan->spare = spare;
  plan->grid = (int)(items_max < p_target ? items_max : p_target);
  if (plan->grid < 1) plan->grid = 1;
  plan->smem = k.smem;
  // a chunk must stream enough keys to amortise its fixed costs (tensor-core kernel: two stages)
  plan->min_chunk = mma ? 128 : 32;
  // an automatic chunk size and groups (b, kv head, row block) that fit the GPU in one wave
  // of clusters of at least two CTAs, about two CTAs per SM: one cluster per group, the
  // largest that fits (its CTAs share the group's keys evenly and merge on chip)
  plan->cluster = 0;
  if (mma && !q8 && split == 0) {
    const long long groups = (long long)B * U;
    for (int cs = kMaxCluster; cs >= 2; cs /= 2) {
      if (groups * cs * 5 < (long long)sms * 8) break;
      if (groups <= active_clusters(device, D, cs)) {
        plan->cluster = cs;
        plan->grid = (int)(groups * cs);
        plan->smem = D == 64 ? cluster_smem<64>() : cluster_smem<128>();
        break;
      }
    }
  }
  // L2 warm-up before the wait for the previous kernel, in units of 64 rows of K and V of
  // each CTA's first chunk. One row block per kv head: up to 16 units while the requests of
  // the whole grid stay within 90% of L2; past that, lines warmed last evict lines warmed
  // first before they are read. Measured on the 3B-style layer at 32k (296 CTAs, chunks of
  // 14 units): 16 units (the whole chunk, about 134 MB) 24.1 us, 13 23.8, 12 (116 MB) 23.5,
  // 11 23.7, 8 24.0; B = 2 at 16k 26.1 / 25.7 / 25.4 / 25.3 / -. The bound takes every
  // CTA's chunk as at least that long (the lengths live on the device); a batch whose keys
  // all fit in L2 can lose a little (the ragged batch of 8: 26.1 -> 26.3 us). Several row
  // blocks per kv head read each tile more than once and warm 4 units (the 6-token verify:
  // 27.8 us without, 27.5 with 4, 29.9 with 16).
  {
    const long long unit = 2LL * 64 * (q8 ? D + 4 : (long long)D * (dtype == TD_F32 ? 4 : 2));
    const long long l2 = device_l2_bytes(device);
    const long long warm = RB == 1 ? (l2 * 9 / 10) / ((long long)plan->grid * unit) : 4;
    plan->warm = (int)(warm < 1 ? 1 : warm > 16 ? 16 : warm);
  }
  // completion counters, one per (b, kv head, row block), then as many counts of finished
  // slice merges, then the fused step's read count
  plan->counters_n = (int)(2LL * B * U);
  const size_t counters = align256(((size_t)plan->counters_n + 1) * sizeof(int));
  plan->off_part = counters;
  plan->bytes = plan->off_part + align256((size_t)B * U * ns * part_block_floats(R, D) * sizeof(float));
  return TD_OK;
}

cudaError_t launch_split(td_dtype dtype, int D, const SplitPlan &plan, const SplitParams &p, cudaStream_t stream) {
  cudaError_t e;
  if (plan.q8) {
    e = D == 64 ? launch_q8<64>(p, plan.grid, plan.smem, plan.spare, stream)
                : launch_q8<128>(p, plan.grid, plan.smem, plan.spare, stream);
  } else if (plan.cluster > 0) {
    e = D == 64 ? launch_cluster<64>(p, plan.grid, plan.cluster, stream)
                : launch_cluster<128>(p, plan.grid, plan.cluster, stream);
  } else {
    const KernelRef k = pick(dtype, D, plan.mma, plan.RP);
    if (k.fn == nullptr) return cudaErrorInvalidValue;
    e = k.launch(p, plan.grid, plan.smem, stream);
  }
  if (e != cudaSuccess) {
    cudaGetLastError();  // clear a launch error so it is reported once, by this call
    return e;
  }
  return cudaSuccess;
}

}  // namespace td
