// api.cu -- the C ABI declared in include/spmv.h: handle life cycle,
// device-memory pool, validation read-back, format selection, conversion and
// SpMV dispatch. All arithmetic on the matrix runs in the CUDA kernels of
// stats.cu, convert.cu and spmv_kernels.cu.
#include <algorithm>
#include <atomic>
#include <climits>
#include <cstring>
#include <mutex>
#include <type_traits>
#include <new>
#include <vector>

#include "internal.h"

namespace {

using spmv::DevStats;

// ---------------------------------------------------------------------------
// Process-wide state
// ---------------------------------------------------------------------------
std::atomic<unsigned long long> g_launches{0};
std::atomic<long long> g_memLimit{-1};
std::atomic<long long> g_memInUse{0};
thread_local int g_lastCudaError = 0;

constexpr int kMaxDevices = 64;
std::mutex g_poolMu;
cudaMemPool_t g_pools[kMaxDevices] = {};
int g_smCount[kMaxDevices] = {};

int record(cudaError_t e) {
  if (e != cudaSuccess) {
    g_lastCudaError = (int)e;
    return e == cudaErrorMemoryAllocation ? SPMV_ERR_ALLOC : SPMV_ERR_CUDA;
  }
  return SPMV_OK;
}

#define SPMV_TRY(expr)            \
  do {                            \
    int st_ = (expr);             \
    if (st_ != SPMV_OK) return st_; \
  } while (0)

// A library-private stream-ordered pool per device, kept at full size
// between uses (release threshold = max), so repeated create/convert/destroy
// cycles do not return memory to the driver.
int get_pool(int dev, cudaMemPool_t* out) {
  if (dev < 0 || dev >= kMaxDevices) return SPMV_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lk(g_poolMu);
  if (!g_pools[dev]) {
    cudaMemPoolProps props;
    std::memset(&props, 0, sizeof(props));
    props.allocType = cudaMemAllocationTypePinned;
    props.handleTypes = cudaMemHandleTypeNone;
    props.location.type = cudaMemLocationTypeDevice;
    props.location.id = dev;
    cudaMemPool_t pool;
    SPMV_TRY(record(cudaMemPoolCreate(&pool, &props)));
    unsigned long long threshold = ~0ull;
    cudaError_t e = cudaMemPoolSetAttribute(pool, cudaMemPoolAttrReleaseThreshold, &threshold);
    if (e != cudaSuccess) {
      cudaMemPoolDestroy(pool);
      return record(e);
    }
    g_pools[dev] = pool;
  }
  *out = g_pools[dev];
  return SPMV_OK;
}

struct Buf {
  void* p;
  size_t bytes;
};

struct DeviceGuard {
  int prev = -1;
  bool changed = false;
  int set(int dev) {
    SPMV_TRY(record(cudaGetDevice(&prev)));
    if (prev != dev) {
      SPMV_TRY(record(cudaSetDevice(dev)));
      changed = true;
    }
    return SPMV_OK;
  }
  ~DeviceGuard() {
    if (changed) cudaSetDevice(prev);
  }
};

// Device memory (or managed memory) on device `dev`; anything else (host,
// pageable, another device) is rejected before a kernel could touch it.
// Page-locked host buffer for the statistics read-back, one per host thread
// (allocated on the thread's first create, kept until exit), so that the
// copy is a plain DMA.
DevStats* pinned_stats_buffer() {
  thread_local DevStats* buf = nullptr;
  if (!buf) {
    void* p = nullptr;
    if (cudaMallocHost(&p, sizeof(DevStats)) != cudaSuccess) {
      cudaGetLastError();
      return nullptr;
    }
    buf = static_cast<DevStats*>(p);
  }
  return buf;
}

int check_device_ptr(const void* p, int dev) {
  cudaPointerAttributes a;
  cudaError_t e = cudaPointerGetAttributes(&a, p);
  if (e != cudaSuccess) {
    cudaGetLastError();  // clear the sticky-free error state of this query
    return SPMV_ERR_INVALID_ARG;
  }
  if (a.type == cudaMemoryTypeManaged) return SPMV_OK;
  if (a.type == cudaMemoryTypeDevice && a.device == dev) return SPMV_OK;
  return SPMV_ERR_INVALID_ARG;
}

}  // namespace

namespace spmv {
void note_launches(int n) { g_launches.fetch_add((unsigned long long)n, std::memory_order_relaxed); }

int record_cuda(cudaError_t e) { return record(e); }

int num_sms() {
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= kMaxDevices) return 152;
  if (!g_smCount[dev]) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      n = 152;
    g_smCount[dev] = n;
  }
  return g_smCount[dev];
}
}  // namespace spmv

// ---------------------------------------------------------------------------
// Handle
// ---------------------------------------------------------------------------
struct spmv_handle_s {
  int device = 0;
  cudaMemPool_t pool = nullptr;
  cudaStream_t lastStream = nullptr;
  int R = 0, C = 0, Z = 0;
  const int* rowPtrs = nullptr;
  const int* colIdx = nullptr;
  const void* value = nullptr;  // float or double (f64)
  bool f64 = false;             // 8-byte values and vectors
  spmv_stats stats;
  std::vector<unsigned> histExact;  // exact row-length counts for len < kExactLenBins

  // CSR: nnz-balanced split, one warp per kCsrChunk nonzeros (computed at creation)
  int nChunks = 0;
  spmv::CsrChunkDesc* chunkDesc = nullptr;  // one record per kCsrChunk nonzeros
  std::vector<Buf> csrBufs;

  // COO (shares colIdx/value with the caller's CSR arrays)
  bool hasCoo = false;
  int* cooRow = nullptr;
  std::vector<Buf> cooBufs;

  // ELL
  bool hasEll = false;
  int ellK = 0;
  int* ellCol = nullptr;
  void* ellVal = nullptr;
  int* ellNnz = nullptr;
  std::vector<Buf> ellBufs;

  // HYB
  bool hasHyb = false;
  int hybK = 0;
  int hybCooN = 0;
  int* hybCol = nullptr;
  void* hybVal = nullptr;
  int* hybNnz = nullptr;
  int* hybCooRow = nullptr;
  int* hybCooCol = nullptr;
  void* hybCooVal = nullptr;
  std::vector<Buf> hybBufs;

  // JDS
  bool hasJds = false;
  int jdsMaxLen = 0;
  int jdsTSplit = 0;
  int jdsWTail = 0;
  std::vector<int> jdsIpHost;  // iterPtr[0 .. jdsTSplit], from the length histogram
  int* jdsPerm = nullptr;
  int* jdsIterPtr = nullptr;
  int* jdsCol = nullptr;
  void* jdsVal = nullptr;
  std::vector<Buf> jdsBufs;

  // SELL (sectioned ELL, the JDS variant)
  bool hasSell = false;
  int sellS = 0;
  int sellW0 = 0;          // widest section
  long long sellSlots = 0;
  int sellNItems = 0;
  int* sellPerm = nullptr;
  int* sellSecPtr = nullptr;
  int* sellCol = nullptr;
  void* sellVal = nullptr;
  spmv::SellItem* sellItems = nullptr;
  std::vector<Buf> sellBufs;

  // XBLOCK (nonzeros grouped by column chunk of x)
  bool hasXb = false;
  int xbB = 0;
  int xbNch = 0;
  long long xbSlots = -1;  // read from the device on first export
  int* xbChunkPtr = nullptr;
  int* xbRow = nullptr;
  unsigned short* xbCol = nullptr;
  void* xbVal = nullptr;
  std::vector<Buf> xbBufs;

  int alloc(size_t bytes, cudaStream_t s, void** out, std::vector<Buf>& list) {
    *out = nullptr;
    if (bytes == 0) return SPMV_OK;
    const long long lim = g_memLimit.load();
    const long long now = g_memInUse.fetch_add((long long)bytes) + (long long)bytes;
    if (lim >= 0 && now > lim) {
      g_memInUse.fetch_sub((long long)bytes);
      return SPMV_ERR_ALLOC;
    }
    void* p = nullptr;
    cudaError_t e = cudaMallocFromPoolAsync(&p, bytes, pool, s);
    if (e != cudaSuccess) {
      g_memInUse.fetch_sub((long long)bytes);
      return record(e);
    }
    list.push_back({p, bytes});
    *out = p;
    return SPMV_OK;
  }

  void release(std::vector<Buf>& list, cudaStream_t s) {
    for (const Buf& b : list) {
      cudaFreeAsync(b.p, s);
      g_memInUse.fetch_sub((long long)b.bytes);
    }
    list.clear();
  }

  // width(t) = number of rows longer than t, exact for t < kExactLenBins
  long long width_at(int t) const {
    long long le = 0;
    for (int L = 0; L <= t && L < spmv::kExactLenBins; ++L) le += histExact[L];
    return (long long)R - le;
  }
};

namespace {

// n values of the handle's value type (4 or 8 bytes)
int alloc_values(spmv_handle h, long long n, cudaStream_t s, void** out, std::vector<Buf>& list) {
  return h->alloc((size_t)n * (h->f64 ? sizeof(double) : sizeof(float)), s, out, list);
}

// Calls f(T{}) with T = the handle's value type; f returns a cudaError_t.
template <class F>
cudaError_t with_type(const spmv_handle_s* h, F&& f) {
  return h->f64 ? f(double{}) : f(float{});
}

template <class T>
const T* cval(const void* p) {
  return static_cast<const T*>(p);
}
template <class T>
T* val(void* p) {
  return static_cast<T*>(p);
}

template <class T>
int alloc_typed(spmv_handle h, long long n, cudaStream_t s, T** out, std::vector<Buf>& list) {
  void* p = nullptr;
  int st = h->alloc((size_t)n * sizeof(T), s, &p, list);
  *out = static_cast<T*>(p);
  return st;
}

// Format choice ("[CUDA performance tuning] SpMV storage format selection and
// performance comparison", section 4.3). The page's comparison operators are
// lost; the reading: longest <= 2*mean -> ELL, else mean < 10 -> COO, else
// HYB when longest > 5*mean, otherwise CSR. Two rules of ours around it,
// from measurements on GB300 (the fastest format of each workload type):
//  - compulsory SpMV bytes below kSmallMatrixBytes -> CSR, first: such a
//    matrix is bound by dependent memory round trips, not bandwidth, and the
//    nnz-balanced CSR kernel has the fewest (4096 x 4096 with 8 per row:
//    CSR 6.8 us, ELL 10.9 us);
//  - in the HYB case, scattered columns (gatherLines >= kScatteredLines: the
//    sampled distinct 128-byte lines of x among 32 consecutive nonzeros) ->
//    XBLOCK, whose gathers come from shared memory ("Introduction to sparse
//    computing and performance bottleneck location", x-blocking): 2M rows of
//    10-20 random columns plus 200 rows of 1000-5000, XBLOCK 113 us against
//    HYB 120 us.
constexpr double kSmallMatrixBytes = 4194304.0;
constexpr double kScatteredLines = 16.0;
int select_format(long long R, long long C, long long Z, long long maxLen, double gatherLines) {
  const double mean = R > 0 ? (double)Z / (double)R : 0.0;
  if (8.0 * (double)Z + 12.0 * (double)R + 4.0 * (double)C < kSmallMatrixBytes) return SPMV_CSR;
  if ((double)maxLen <= 2.0 * mean) return SPMV_ELL;
  if (mean < 10.0) return SPMV_COO;
  if ((double)maxLen > 5.0 * mean) return gatherLines >= kScatteredLines ? SPMV_XBLOCK : SPMV_HYB;
  return SPMV_CSR;
}

// Automatic HYB width: smallest L with 100 * #{len <= L} >= 99 * R (section
// 4.1 of the same page keeps the 99% of rows of length 10-20 whole in an ELL
// part of width 20). Beyond the exact histogram the log2 bins give an upper
// bound, capped at the longest row.
int auto_hyb_width(const spmv_handle_s* h) {
  const long long R = h->R;
  if (R == 0) return 0;
  long long cum = 0;
  for (int L = 0; L < spmv::kExactLenBins && L <= h->stats.max_len; ++L) {
    cum += h->histExact[L];
    if (100 * cum >= 99 * R) return L;
  }
  // remaining rows are at least kExactLenBins long; walk the log2 bins
  long long cumLog = 0;
  for (int b = 0; b < 33; ++b) {
    cumLog += h->stats.hist_log2[b];
    if (100 * cumLog >= 99 * R) {
      long long upper = b == 0 ? 0 : (1LL << b) - 1;
      if (upper > h->stats.max_len) upper = h->stats.max_len;
      return (int)upper;
    }
  }
  return (int)h->stats.max_len;
}

// ELL/HYB slot budget: numRows*K within int32 and at most 4*nnz + numRows.
bool ell_fits(long long R, long long K, long long Z) {
  const long long slots = R * K;
  return slots <= (long long)INT_MAX && slots <= 4 * Z + R;
}

int check_handle(spmv_handle h) { return h ? SPMV_OK : SPMV_ERR_INVALID_ARG; }

}  // namespace

// ---------------------------------------------------------------------------
// Exported functions
// ---------------------------------------------------------------------------
extern "C" {

namespace {
int create_impl(spmv_handle* out, int32_t numRows, int32_t numCols, int32_t nnz,
                const int32_t* d_rowPtrs, const int32_t* d_colIdx, const void* d_value, bool f64,
                void* stream) {
  if (!out) return SPMV_ERR_INVALID_ARG;
  *out = nullptr;
  if (numRows < 0 || numCols < 0 || nnz < 0 || !d_rowPtrs) return SPMV_ERR_INVALID_ARG;
  if (nnz > 0 && (!d_colIdx || !d_value)) return SPMV_ERR_INVALID_ARG;
  if (nnz > 0 && numCols == 0) return SPMV_ERR_COL_OUT_OF_RANGE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int dev = 0;
  SPMV_TRY(record(cudaGetDevice(&dev)));
  SPMV_TRY(check_device_ptr(d_rowPtrs, dev));
  if (nnz > 0) {
    SPMV_TRY(check_device_ptr(d_colIdx, dev));
    SPMV_TRY(check_device_ptr(d_value, dev));
  }
  spmv_handle h = new (std::nothrow) spmv_handle_s();
  if (!h) return SPMV_ERR_ALLOC;
  h->device = dev;
  h->R = numRows;
  h->C = numCols;
  h->Z = nnz;
  h->rowPtrs = d_rowPtrs;
  h->colIdx = d_colIdx;
  h->value = d_value;
  h->f64 = f64;
  h->lastStream = s;
  int st = get_pool(dev, &h->pool);
  std::vector<Buf> tmp;
  auto fail = [&](int code) {
    h->release(tmp, s);
    h->release(h->csrBufs, s);
    delete h;
    return code;
  };
  if (st != SPMV_OK) return fail(st);
  DevStats* hst = pinned_stats_buffer();
  if (!hst) return fail(SPMV_ERR_ALLOC);
  // One allocation, zeroed by one memset: the statistics record (its work
  // area, a multiple of 256 bytes) followed by the nnz-balanced split for the
  // CSR kernel, whose masks and flags the statistics pass ORs into zeroed
  // records (it checks bounds, so it stays in bounds even if validation
  // fails). Both stay with the handle.
  h->nChunks = (int)(((long long)nnz + spmv::kCsrChunk - 1) / spmv::kCsrChunk);
  const size_t statsBytes = spmv::stats_work_bytes(numRows, nnz, d_colIdx);
  const size_t zeroBytes = statsBytes + sizeof(spmv::CsrChunkDesc) * (size_t)h->nChunks;
  void* work = nullptr;
  st = h->alloc(zeroBytes, s, &work, h->csrBufs);
  if (st != SPMV_OK) return fail(st);
  st = record(cudaMemsetAsync(work, 0, zeroBytes, s));
  if (st != SPMV_OK) return fail(st);
  h->chunkDesc = h->nChunks > 0 ? reinterpret_cast<spmv::CsrChunkDesc*>(
                                      static_cast<char*>(work) + statsBytes)
                                : nullptr;
  st = record(spmv::launch_stats(numRows, numCols, nnz, d_rowPtrs, d_colIdx, work, h->nChunks,
                                 h->chunkDesc, s));
  if (st != SPMV_OK) return fail(st);
  st = record(cudaMemcpyAsync(hst, work, sizeof(DevStats), cudaMemcpyDeviceToHost, s));
  if (st != SPMV_OK) return fail(st);
  st = record(cudaStreamSynchronize(s));
  if (st != SPMV_OK) return fail(st);
  const unsigned errs = spmv::stats_errors(*hst);
  if (errs & (spmv::kErrRowPtrStart | spmv::kErrRowPtrDecrease | spmv::kErrRowPtrEnd))
    return fail(SPMV_ERR_BAD_ROWPTRS);
  if (errs & spmv::kErrColRange) return fail(SPMV_ERR_COL_OUT_OF_RANGE);

  spmv_stats& S = h->stats;
  std::memset(&S, 0, sizeof(S));
  S.num_rows = numRows;
  S.num_cols = numCols;
  S.nnz = nnz;
  S.max_len = hst->maxLen;
  S.min_len = numRows > 0 ? spmv::stats_min_len(*hst) : 0;
  S.empty_rows = hst->emptyRows;
  S.sum_sq_len = (int64_t)hst->sumSq;
  S.mean_len = numRows > 0 ? (double)nnz / (double)numRows : 0.0;
  if (numRows > 0) {
    const long double Rl = numRows, Zl = nnz;
    const long double num = Rl * (long double)hst->sumSq - Zl * Zl;
    S.var_len = (double)(num / Rl / Rl);
  }
  for (int b = 0; b < 33; ++b) S.hist_log2[b] = (int64_t)hst->histLog2[b];
  for (int L = 0; L < spmv::kExactLenBins; ++L) {
    // bin 0: len 0; bin b >= 1: len in [2^(b-1), 2^b)
    const int b = L == 0 ? 0 : 32 - __builtin_clz((unsigned)L);
    S.hist_log2[b] += hst->histExact[L];
  }
  S.imbalance_thread = S.mean_len > 0 ? (double)S.max_len / S.mean_len : 0.0;
  if (numRows > 0 && nnz > 0) {
    const double groups = (double)((numRows + 31) / 32);
    S.imbalance_warp = (double)hst->maxWarpNnz / ((double)nnz / groups);
  }
  h->histExact.assign(hst->histExact, hst->histExact + spmv::kExactLenBins);
  S.gather_lines = hst->gatherSets ? (double)hst->gatherLines / (double)hst->gatherSets : 0.0;
  S.auto_format = select_format(numRows, numCols, nnz, S.max_len, S.gather_lines);
  S.auto_hyb_width = auto_hyb_width(h);
  h->release(tmp, s);
  *out = h;
  return SPMV_OK;
}
}  // namespace

int spmv_create_csr(spmv_handle* out, int32_t numRows, int32_t numCols, int32_t nnz,
                    const int32_t* d_rowPtrs, const int32_t* d_colIdx, const float* d_value,
                    void* stream) {
  return create_impl(out, numRows, numCols, nnz, d_rowPtrs, d_colIdx, d_value, false, stream);
}

int spmv_create_csr_f64(spmv_handle* out, int32_t numRows, int32_t numCols, int32_t nnz,
                        const int32_t* d_rowPtrs, const int32_t* d_colIdx, const double* d_value,
                        void* stream) {
  return create_impl(out, numRows, numCols, nnz, d_rowPtrs, d_colIdx, d_value, true, stream);
}

int spmv_convert_coo(spmv_handle h, void* stream) {
  SPMV_TRY(check_handle(h));
  DeviceGuard g;
  SPMV_TRY(g.set(h->device));
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  h->lastStream = s;
  h->release(h->cooBufs, s);
  h->hasCoo = false;
  SPMV_TRY(alloc_typed(h, h->Z, s, &h->cooRow, h->cooBufs));
  SPMV_TRY(record(spmv::launch_expand_rows(h->R, h->Z, h->rowPtrs, h->chunkDesc, h->cooRow, s)));
  h->hasCoo = true;
  return SPMV_OK;
}

int spmv_convert_ell(spmv_handle h, void* stream) {
  SPMV_TRY(check_handle(h));
  DeviceGuard g;
  SPMV_TRY(g.set(h->device));
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  h->lastStream = s;
  const long long K = h->stats.max_len;
  if (!ell_fits(h->R, K, h->Z)) return SPMV_ERR_TOO_LARGE;
  h->release(h->ellBufs, s);
  h->hasEll = false;
  const long long slots = (long long)h->R * K;
  SPMV_TRY(alloc_typed(h, slots, s, &h->ellCol, h->ellBufs));
  SPMV_TRY(alloc_values(h, slots, s, &h->ellVal, h->ellBufs));
  SPMV_TRY(alloc_typed(h, h->R, s, &h->ellNnz, h->ellBufs));
  SPMV_TRY(record(with_type(h, [&](auto tag) {
    using T = decltype(tag);
    return spmv::launch_csr_to_ell<T>(h->R, (int)K, h->rowPtrs, h->colIdx, cval<T>(h->value),
                                      h->ellCol, val<T>(h->ellVal), h->ellNnz, s);
  })));
  h->ellK = (int)K;
  h->hasEll = true;
  return SPMV_OK;
}

int spmv_convert_hyb(spmv_handle h, int32_t ellWidth, void* stream) {
  SPMV_TRY(check_handle(h));
  if (ellWidth < 0) return SPMV_ERR_INVALID_ARG;
  DeviceGuard g;
  SPMV_TRY(g.set(h->device));
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  h->lastStream = s;
  long long K = ellWidth > 0 ? ellWidth : h->stats.auto_hyb_width;
  if (K > h->stats.max_len) K = h->stats.max_len;
  if (!ell_fits(h->R, K, h->Z)) return SPMV_ERR_TOO_LARGE;
  h->release(h->hybBufs, s);
  h->hasHyb = false;
  const long long R = h->R;
  const long long slots = R * K;
  SPMV_TRY(alloc_typed(h, slots, s, &h->hybCol, h->hybBufs));
  SPMV_TRY(alloc_values(h, slots, s, &h->hybVal, h->hybBufs));
  SPMV_TRY(alloc_typed(h, R, s, &h->hybNnz, h->hybBufs));
  SPMV_TRY(record(with_type(h, [&](auto tag) {
    using T = decltype(tag);
    return spmv::launch_csr_to_ell<T>(h->R, (int)K, h->rowPtrs, h->colIdx, cval<T>(h->value),
                                      h->hybCol, val<T>(h->hybVal), h->hybNnz, s);
  })));
  // COO part size: nnz - sum_r min(len_r, K), exact from the histogram when
  // K is below the exact range (longer rows then all keep K entries).
  long long tail = -1;
  if (K < spmv::kExactLenBins) {
    long long kept = 0, counted = 0;
    for (int L = 0; L < spmv::kExactLenBins; ++L) {
      kept += (long long)h->histExact[L] * (L < K ? L : K);
      counted += h->histExact[L];
    }
    kept += (R - counted) * K;
    tail = (long long)h->Z - kept;
  }
  if (tail == 0) {  // every row fits in the ELL part: no COO part
    h->hybK = (int)K;
    h->hybCooN = 0;
    h->hasHyb = true;
    return SPMV_OK;
  }
  std::vector<Buf> tmp;
  int* tailPtr = nullptr;
  int* scratch = nullptr;
  auto done = [&](int code) {
    h->release(tmp, s);
    return code;
  };
  int st = alloc_typed(h, R + 1, s, &tailPtr, tmp);
  if (st == SPMV_OK) st = alloc_typed(h, (long long)spmv::scan_scratch_ints(R), s, &scratch, tmp);
  if (st == SPMV_OK) st = record(spmv::launch_tail_scan(h->R, (int)K, h->rowPtrs, tailPtr, scratch, s));
  if (st != SPMV_OK) return done(st);
  if (tail < 0) {
    int t = 0;
    st = record(cudaMemcpyAsync(&t, tailPtr + R, sizeof(int), cudaMemcpyDeviceToHost, s));
    if (st == SPMV_OK) st = record(cudaStreamSynchronize(s));
    if (st != SPMV_OK) return done(st);
    tail = t;
  }
  st = alloc_typed(h, tail, s, &h->hybCooRow, h->hybBufs);
  if (st == SPMV_OK) st = alloc_typed(h, tail, s, &h->hybCooCol, h->hybBufs);
  if (st == SPMV_OK) st = alloc_values(h, tail, s, &h->hybCooVal, h->hybBufs);
  if (st == SPMV_OK && tail > 0)
    st = record(with_type(h, [&](auto tag) {
      using T = decltype(tag);
      return spmv::launch_hyb_tail_copy<T>(h->R, (int)K, h->rowPtrs, h->colIdx,
                                           cval<T>(h->value), tailPtr, h->hybCooRow,
                                           h->hybCooCol, val<T>(h->hybCooVal), s);
    }));
  if (st != SPMV_OK) return done(st);
  h->hybK = (int)K;
  h->hybCooN = (int)tail;
  h->hasHyb = true;
  return done(SPMV_OK);
}

int spmv_convert_jds(spmv_handle h, void* stream) {
  SPMV_TRY(check_handle(h));
  DeviceGuard g;
  SPMV_TRY(g.set(h->device));
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  h->lastStream = s;
  h->release(h->jdsBufs, s);
  h->hasJds = false;
  const int L = (int)h->stats.max_len;
  SPMV_TRY(alloc_typed(h, h->R, s, &h->jdsPerm, h->jdsBufs));
  SPMV_TRY(alloc_typed(h, (long long)L + 1, s, &h->jdsIterPtr, h->jdsBufs));
  // padded so that the SpMV kernel's aligned 16-byte reads stay inside
  SPMV_TRY(alloc_typed(h, (long long)h->Z + spmv::kJdsPad, s, &h->jdsCol, h->jdsBufs));
  SPMV_TRY(alloc_values(h, (long long)h->Z + spmv::kJdsPad, s, &h->jdsVal, h->jdsBufs));
  // iterPtr from the exact length histogram when every row is shorter than
  // kExactLenBins: iterPtr[t+1] = iterPtr[t] + #{rows longer than t}
  std::vector<int> hostIp;
  if (L > 0 && L < spmv::kExactLenBins) {
    hostIp.assign((size_t)L + 1, 0);
    long long le = 0, acc = 0;
    for (int t = 0; t < L; ++t) {
      le += h->histExact[t];
      acc += (long long)h->R - le;
      hostIp[(size_t)t + 1] = (int)acc;
    }
  }
  std::vector<Buf> tmp;
  void* scratch = nullptr;
  int st = h->alloc(spmv::jds_sort_scratch_bytes(h->R, L), s, &scratch, tmp);
  if (st == SPMV_OK)
    st = record(with_type(h, [&](auto tag) {
      using T = decltype(tag);
      // rows longer than kJdsCoop: exact from the length histogram (kJdsCoop < kExactLenBins)
      const int wLong = (int)h->width_at(spmv::kJdsCoop);
      return spmv::launch_jds_build<T>(h->R, L, wLong, h->rowPtrs, h->colIdx, cval<T>(h->value),
                                       h->jdsPerm, h->jdsIterPtr, h->jdsCol, val<T>(h->jdsVal),
                                       scratch, hostIp.empty() ? nullptr : hostIp.data(), s);
    }));
  h->release(tmp, s);
  if (st != SPMV_OK) return st;
  // Row-parallel part: the leading diagonals at least min(kJdsSplitMinWidth,
  // width(0)) wide, at most kJdsSplitMaxDiag of them (widths are exact from
  // the histogram there).
  const long long w0 = h->width_at(0);
  const long long thr = w0 < spmv::kJdsSplitMinWidth ? w0 : spmv::kJdsSplitMinWidth;
  int tSplit = 0;
  const int cap = L < spmv::kJdsSplitMaxDiag ? L : spmv::kJdsSplitMaxDiag;
  while (tSplit < cap && thr > 0 && h->width_at(tSplit) >= thr) ++tSplit;
  h->jdsTSplit = tSplit;
  h->jdsWTail = tSplit < L ? (int)h->width_at(tSplit) : 0;
  h->jdsIpHost.assign((size_t)tSplit + 1, 0);
  for (int t = 0; t < tSplit; ++t)
    h->jdsIpHost[(size_t)t + 1] = h->jdsIpHost[(size_t)t] + (int)h->width_at(t);
  h->jdsMaxLen = L;
  h->hasJds = true;
  return SPMV_OK;
}

int spmv_convert_sell(spmv_handle h, int32_t sectionRows, void* stream) {
  SPMV_TRY(check_handle(h));
  if (sectionRows < 0) return SPMV_ERR_INVALID_ARG;
  const int S = sectionRows > 0 ? sectionRows : spmv::kSellDefaultRows;
  DeviceGuard g;
  SPMV_TRY(g.set(h->device));
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  h->lastStream = s;
  h->release(h->sellBufs, s);
  h->hasSell = false;
  const long long R = h->R;
  const int L = (int)h->stats.max_len;
  const long long nsec = (R + S - 1) / S;
  const long long budget = 4LL * h->Z + R < INT32_MAX ? 4LL * h->Z + R : INT32_MAX;
  auto section_rows = [&](long long k) { return R - k * S < S ? R - k * S : (long long)S; };
  // Section widths (length of each section's first sorted row). With every
  // row shorter than kExactLenBins they follow from the exact length
  // histogram, before any device work: the size check comes first and the
  // section offsets are scanned on the device. Otherwise they are computed on
  // the device after the sort and read back (one synchronisation).
  const bool fromHist = L < spmv::kExactLenBins;
  // sections [k0, k1) of width w, in section order (widths only shrink)
  struct WidthRun {
    long long k0, k1;
    int w;
  };
  std::vector<WidthRun> runs;
  long long slots = 0;
  // rows of sections [k0, k1): S each, the last section possibly fewer
  auto rows_of = [&](long long k0, long long k1) {
    return k1 <= k0 ? 0 : (k1 - k0 - 1) * S + section_rows(k1 - 1);
  };
  if (fromHist) {
    // one run per length present: the sections whose first sorted row has
    // that length (O(longest row) host work, not O(sections))
    long long pos = 0;  // sorted positions [pos, pos + count) have length len
    for (int len = L; len >= 0 && pos < R; --len) {
      const long long c = h->histExact[len];
      const long long k0 = (pos + S - 1) / S;
      long long k1 = (pos + c + S - 1) / S;  // sections with k * S < pos + c
      if (k1 > nsec) k1 = nsec;
      if (k1 > k0) {
        runs.push_back({k0, k1, len});
        slots += rows_of(k0, k1) * len;
      }
      pos += c;
    }
    if (slots > budget) return SPMV_ERR_TOO_LARGE;
  }
  std::vector<Buf> tmp;
  auto fail = [&](int code) {
    h->release(tmp, s);
    h->release(h->sellBufs, s);
    return code;
  };
  int st = alloc_typed(h, R, s, &h->sellPerm, h->sellBufs);
  if (st == SPMV_OK) st = alloc_typed(h, nsec + 1, s, &h->sellSecPtr, h->sellBufs);
  // the slot arrays before the scratch when their size is known: the pool
  // then reuses the previous conversion's blocks for them instead of cutting
  // the scratch out of one and mapping new memory (a 27-point stencil's
  // repeated conversion: host time 120-570 us before, about 30 us after;
  // 480-860 us -> 377 us on the device)
  if (fromHist) {
    if (st == SPMV_OK) st = alloc_typed(h, slots, s, &h->sellCol, h->sellBufs);
    if (st == SPMV_OK) st = alloc_values(h, slots, s, &h->sellVal, h->sellBufs);
  }
  void* scratch = nullptr;
  if (st == SPMV_OK) st = h->alloc(spmv::sell_scratch_bytes(h->R, L, nsec), s, &scratch, tmp);
  if (st == SPMV_OK)
    st = record(spmv::launch_sell_sort(h->R, L, h->rowPtrs, h->sellPerm, scratch, s));
  if (st != SPMV_OK) return fail(st);
  if (fromHist) {
    st = record(spmv::launch_sell_offsets(h->R, S, L, nsec, h->rowPtrs, h->sellPerm,
                                          h->sellSecPtr, scratch, s));
  } else {
    int* dW = nullptr;
    std::vector<int> width((size_t)nsec, 0);
    st = alloc_typed(h, nsec, s, &dW, tmp);
    if (st == SPMV_OK)
      st = record(spmv::launch_sell_widths(h->R, S, (int)nsec, h->rowPtrs, h->sellPerm, dW, s));
    if (st == SPMV_OK)
      st = record(cudaMemcpyAsync(width.data(), dW, sizeof(int) * (size_t)nsec,
                                  cudaMemcpyDeviceToHost, s));
    if (st == SPMV_OK) st = record(cudaStreamSynchronize(s));
    if (st != SPMV_OK) return fail(st);
    std::vector<int> secPtr((size_t)nsec + 1, 0);
    for (long long k = 0; k < nsec; ++k) {
      secPtr[(size_t)k] = (int)slots;
      slots += section_rows(k) * width[(size_t)k];
      if (slots > budget) return fail(SPMV_ERR_TOO_LARGE);  // int32 offsets, ELL's budget
      if (runs.empty() || runs.back().w != width[(size_t)k])
        runs.push_back({k, k + 1, width[(size_t)k]});
      else
        runs.back().k1 = k + 1;
    }
    secPtr[(size_t)nsec] = (int)slots;
    st = record(cudaMemcpyAsync(h->sellSecPtr, secPtr.data(), sizeof(int) * secPtr.size(),
                                cudaMemcpyHostToDevice, s));
  }
  if (!fromHist) {
    if (st == SPMV_OK) st = alloc_typed(h, slots, s, &h->sellCol, h->sellBufs);
    if (st == SPMV_OK) st = alloc_values(h, slots, s, &h->sellVal, h->sellBufs);
  }
  if (st == SPMV_OK && slots > 0)
    st = record(with_type(h, [&](auto tag) {
      using T = decltype(tag);
      return spmv::launch_sell_scatter<T>(h->R, S, (int)h->stats.max_len, h->rowPtrs,
                                          h->colIdx, cval<T>(h->value),
                                          scratch, h->sellSecPtr, (int)slots, h->sellCol,
                                          val<T>(h->sellVal), s);
    }));
  if (st != SPMV_OK) return fail(st);
  // tail work items of the sections wider than kSellMainSlots (a prefix)
  std::vector<spmv::SellItem> items;
  const int rowsPerItem = 32;  // one row per lane
  for (const WidthRun& run : runs) {
    if (run.w <= spmv::kSellMainSlots) break;  // widths only shrink
    for (long long k = run.k0; k < run.k1; ++k) {
      const int wk = run.w;
      for (int t0 = spmv::kSellMainSlots; t0 < wk; t0 += spmv::kSellTailSlots) {
        const int t1 = wk - t0 > spmv::kSellTailSlots ? t0 + spmv::kSellTailSlots : wk;
        for (long long j0 = 0; j0 < section_rows(k); j0 += rowsPerItem)
          items.push_back({(int)k, t0, t1, (int)j0});
      }
    }
  }
  if (items.size() > (size_t)INT32_MAX) return fail(SPMV_ERR_TOO_LARGE);
  h->sellItems = nullptr;
  if (!items.empty()) {
    st = alloc_typed(h, (long long)items.size(), s, &h->sellItems, h->sellBufs);
    if (st == SPMV_OK)
      st = record(cudaMemcpyAsync(h->sellItems, items.data(),
                                  sizeof(spmv::SellItem) * items.size(),
                                  cudaMemcpyHostToDevice, s));
    if (st != SPMV_OK) return fail(st);
  }
  h->release(tmp, s);
  h->sellS = S;
  h->sellW0 = runs.empty() ? 0 : runs.front().w;
  h->sellSlots = slots;
  h->sellNItems = (int)items.size();
  h->hasSell = true;
  return SPMV_OK;
}

int spmv_convert_xblock(spmv_handle h, int32_t chunkCols, void* stream) {
  SPMV_TRY(check_handle(h));
  // the SpMV stages B values of x in kXbSmemBytes of shared memory
  const int maxB = spmv::kXbSmemBytes / (h->f64 ? (int)sizeof(double) : (int)sizeof(float));
  if (chunkCols < 0 || chunkCols > maxB) return SPMV_ERR_INVALID_ARG;
  const int B = chunkCols > 0 ? chunkCols : maxB;
  const long long nch = ((long long)h->C + B - 1) / B;
  if (nch > spmv::kXbMaxChunks) return SPMV_ERR_TOO_LARGE;
  const long long bound = (long long)h->Z + 3 * nch;  // slots, padding included
  if (bound > INT32_MAX) return SPMV_ERR_TOO_LARGE;
  DeviceGuard g;
  SPMV_TRY(g.set(h->device));
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  h->lastStream = s;
  h->release(h->xbBufs, s);
  h->hasXb = false;
  std::vector<Buf> tmp;
  auto fail = [&](int code) {
    h->release(tmp, s);
    h->release(h->xbBufs, s);
    return code;
  };
  int st = alloc_typed(h, nch + 1, s, &h->xbChunkPtr, h->xbBufs);
  if (st == SPMV_OK) st = alloc_typed(h, bound, s, &h->xbRow, h->xbBufs);
  if (st == SPMV_OK) st = alloc_typed(h, bound, s, &h->xbCol, h->xbBufs);
  if (st == SPMV_OK) st = alloc_values(h, bound, s, &h->xbVal, h->xbBufs);
  // row of every nonzero, for more than kXbTileChunks chunks: the COO
  // conversion's array when present (fewer chunks decode rows on the fly)
  const int* rowIdx = h->hasCoo ? h->cooRow : nullptr;
  if (st == SPMV_OK && !rowIdx && h->Z > 0 && nch > spmv::kXbTileChunks) {
    int* tmpRow = nullptr;
    st = alloc_typed(h, h->Z, s, &tmpRow, tmp);
    if (st == SPMV_OK)
      st = record(spmv::launch_expand_rows(h->R, h->Z, h->rowPtrs, h->chunkDesc, tmpRow, s));
    rowIdx = tmpRow;
  }
  void* scratch = nullptr;
  if (st == SPMV_OK) st = h->alloc(spmv::xb_scratch_bytes(h->Z, (int)nch), s, &scratch, tmp);
  if (st == SPMV_OK)
    st = record(with_type(h, [&](auto tag) {
      using T = decltype(tag);
      return spmv::launch_xb_build<T>(h->Z, B, (int)nch, h->rowPtrs, h->chunkDesc, h->colIdx,
                                      cval<T>(h->value), rowIdx,
                                      h->stats.gather_lines >= kScatteredLines, h->xbChunkPtr,
                                      h->xbRow, h->xbCol, val<T>(h->xbVal), scratch, s);
    }));
  if (st != SPMV_OK) return fail(st);
  h->release(tmp, s);
  h->xbB = B;
  h->xbNch = (int)nch;
  h->xbSlots = -1;
  h->hasXb = true;
  return SPMV_OK;
}

int spmv_select(spmv_handle h, spmv_format* format, int32_t* ellWidth) {
  SPMV_TRY(check_handle(h));
  if (format) *format = (spmv_format)h->stats.auto_format;
  if (ellWidth) *ellWidth = h->stats.auto_hyb_width;
  return SPMV_OK;
}

}  // extern "C"

namespace {
template <class T>
int run_format(spmv_handle h, spmv_format format, const T* d_x, T* d_y, cudaStream_t s);

int converted(const spmv_handle_s* h, spmv_format format) {
  switch (format) {
    case SPMV_CSR: return SPMV_OK;
    case SPMV_COO: return h->hasCoo ? SPMV_OK : SPMV_ERR_NOT_CONVERTED;
    case SPMV_ELL: return h->hasEll ? SPMV_OK : SPMV_ERR_NOT_CONVERTED;
    case SPMV_HYB: return h->hasHyb ? SPMV_OK : SPMV_ERR_NOT_CONVERTED;
    case SPMV_JDS: return h->hasJds ? SPMV_OK : SPMV_ERR_NOT_CONVERTED;
    case SPMV_SELL: return h->hasSell ? SPMV_OK : SPMV_ERR_NOT_CONVERTED;
    case SPMV_XBLOCK: return h->hasXb ? SPMV_OK : SPMV_ERR_NOT_CONVERTED;
    default: return SPMV_ERR_INVALID_ARG;
  }
}
}  // namespace

namespace {
template <class T>
int run_impl(spmv_handle h, spmv_format format, const T* d_x, T* d_y, void* stream) {
  SPMV_TRY(check_handle(h));
  if (h->f64 != std::is_same<T, double>::value) return SPMV_ERR_INVALID_ARG;  // value type
  if (format == SPMV_AUTO) format = (spmv_format)h->stats.auto_format;
  if (format < SPMV_COO || format > SPMV_XBLOCK || format == SPMV_AUTO)
    return SPMV_ERR_INVALID_ARG;
  if (h->R > 0 && !d_y) return SPMV_ERR_INVALID_ARG;
  if (h->C > 0 && !d_x) return SPMV_ERR_INVALID_ARG;
  if (h->R > 0 && h->C > 0) {
    const char* xb = reinterpret_cast<const char*>(d_x);
    const char* yb = reinterpret_cast<const char*>(d_y);
    if (xb < yb + (size_t)h->R * sizeof(T) && yb < xb + (size_t)h->C * sizeof(T))
      return SPMV_ERR_INVALID_ARG;
  }
  SPMV_TRY(converted(h, format));
  if (h->R == 0) return SPMV_OK;
  DeviceGuard g;
  SPMV_TRY(g.set(h->device));
  SPMV_TRY(check_device_ptr(d_y, h->device));
  if (h->C > 0) SPMV_TRY(check_device_ptr(d_x, h->device));
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  h->lastStream = s;
  return run_format<T>(h, format, d_x, d_y, s);
}
}  // namespace

extern "C" {

int spmv_run(spmv_handle h, spmv_format format, const float* d_x, float* d_y, void* stream) {
  return run_impl<float>(h, format, d_x, d_y, stream);
}

int spmv_run_f64(spmv_handle h, spmv_format format, const double* d_x, double* d_y,
                 void* stream) {
  return run_impl<double>(h, format, d_x, d_y, stream);
}

int spmv_autotune(spmv_handle h, const float* d_x, float* d_y, int32_t reps, spmv_format* best,
                  float* times_ms, void* stream) {
  SPMV_TRY(check_handle(h));
  if (h->f64 || !best || reps < 1 || reps > 1000) return SPMV_ERR_INVALID_ARG;
  if (times_ms)
    for (int f = 0; f < 8; ++f) times_ms[f] = -1.0f;
  DeviceGuard g;
  SPMV_TRY(g.set(h->device));
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaEvent_t ev[2] = {nullptr, nullptr};
  int st = record(cudaEventCreate(&ev[0]));
  if (st == SPMV_OK) st = record(cudaEventCreate(&ev[1]));
  const spmv_format order[] = {SPMV_CSR, SPMV_COO, SPMV_ELL, SPMV_HYB,
                               SPMV_JDS, SPMV_SELL, SPMV_XBLOCK};
  spmv_format fastest = SPMV_CSR;
  float fastestMs = -1.0f;
  std::vector<float> t;
  for (const spmv_format f : order) {
    if (st != SPMV_OK) break;
    if (converted(h, f) != SPMV_OK) continue;
    st = run_impl<float>(h, f, d_x, d_y, stream);  // untimed (checks the arguments too)
    t.clear();
    for (int r = 0; r < reps && st == SPMV_OK; ++r) {
      st = record(cudaEventRecord(ev[0], s));
      if (st == SPMV_OK) st = run_impl<float>(h, f, d_x, d_y, stream);
      if (st == SPMV_OK) st = record(cudaEventRecord(ev[1], s));
      if (st == SPMV_OK) st = record(cudaEventSynchronize(ev[1]));
      float ms = 0.0f;
      if (st == SPMV_OK) st = record(cudaEventElapsedTime(&ms, ev[0], ev[1]));
      if (st == SPMV_OK) t.push_back(ms);
    }
    if (st != SPMV_OK) break;
    std::sort(t.begin(), t.end());
    const float med = t.size() % 2 ? t[t.size() / 2]
                                   : 0.5f * (t[t.size() / 2 - 1] + t[t.size() / 2]);
    if (times_ms) times_ms[f] = med;
    if (fastestMs < 0.0f || med < fastestMs) {
      fastestMs = med;
      fastest = f;
    }
  }
  for (cudaEvent_t e : ev)
    if (e) cudaEventDestroy(e);
  if (st != SPMV_OK) return st;
  h->stats.auto_format = fastest;
  *best = fastest;
  return SPMV_OK;
}

}  // extern "C"

namespace {
// y <- A x + y in a converted format; arguments already checked; T is the
// handle's value type.
template <class T>
int run_format(spmv_handle h, spmv_format format, const T* d_x, T* d_y, cudaStream_t s) {
  const T* value = cval<T>(h->value);
  switch (format) {
    case SPMV_CSR:
      return record(spmv::launch_spmv_csr<T>(h->R, h->Z, h->rowPtrs, h->colIdx, value,
                                             h->chunkDesc, d_x, d_y, s));
    case SPMV_COO:
      return record(spmv::launch_spmv_coo<T>(h->Z, h->cooRow, h->colIdx, value, d_x, d_y, false,
                                             s));
    case SPMV_ELL:
      return record(spmv::launch_spmv_ell<T>(h->R, h->ellK, h->ellCol, cval<T>(h->ellVal), d_x,
                                             d_y, s));
    case SPMV_HYB: {
      bool ellRan = false;
      if (h->hybK > 0) {
        SPMV_TRY(record(spmv::launch_spmv_ell<T>(h->R, h->hybK, h->hybCol, cval<T>(h->hybVal),
                                                 d_x, d_y, s)));
        ellRan = true;
      }
      if (h->hybCooN > 0)
        SPMV_TRY(record(spmv::launch_spmv_coo<T>(h->hybCooN, h->hybCooRow, h->hybCooCol,
                                                 cval<T>(h->hybCooVal), d_x, d_y, ellRan, s)));
      return SPMV_OK;
    }
    case SPMV_JDS:
      return record(spmv::launch_spmv_jds<T>(h->R, h->jdsMaxLen, h->jdsTSplit, h->jdsWTail,
                                             h->jdsIterPtr, h->jdsIpHost.data(), h->jdsPerm,
                                             h->jdsCol, cval<T>(h->jdsVal), d_x, d_y, s));
    case SPMV_SELL:
      if (h->sellSlots == 0) return SPMV_OK;
      return record(spmv::launch_spmv_sell<T>(h->R, h->sellS, (int)h->sellSlots, h->sellSecPtr,
                                              h->sellPerm, h->sellCol, cval<T>(h->sellVal),
                                              h->sellItems, h->sellNItems, d_x, d_y, s));
    case SPMV_XBLOCK:
      return record(spmv::launch_spmv_xb<T>(h->C, h->xbB, h->xbNch, h->xbChunkPtr, h->xbRow,
                                            h->xbCol, cval<T>(h->xbVal), d_x, d_y, s));
    default:
      return SPMV_ERR_INVALID_ARG;
  }
}
}  // namespace

extern "C" {

namespace {
// pinned host copy of the CG state, one per host thread
spmv::CgState* pinned_cg_buffer() {
  thread_local spmv::CgState* buf = nullptr;
  if (!buf) {
    void* p = nullptr;
    if (cudaMallocHost(&p, sizeof(spmv::CgState)) != cudaSuccess) {
      cudaGetLastError();
      return nullptr;
    }
    buf = static_cast<spmv::CgState*>(p);
  }
  return buf;
}
}  // namespace

int spmv_cg_solve(spmv_handle h, spmv_format format, const float* d_y, float* d_x,
                  int32_t maxIter, double tol, spmv_cg_info* info, void* stream) {
  SPMV_TRY(check_handle(h));
  if (!info || maxIter < 0 || !(tol >= 0.0)) return SPMV_ERR_INVALID_ARG;
  if (h->f64) return SPMV_ERR_INVALID_ARG;  // the solver runs on 4-byte values
  if (h->R != h->C) return SPMV_ERR_INVALID_ARG;
  if (format == SPMV_AUTO) format = (spmv_format)h->stats.auto_format;
  SPMV_TRY(converted(h, format));
  std::memset(info, 0, sizeof(*info));
  const long long R = h->R;
  if (R == 0) return SPMV_OK;
  if (!d_y || !d_x) return SPMV_ERR_INVALID_ARG;
  {
    const char* xb = reinterpret_cast<const char*>(d_x);
    const char* yb = reinterpret_cast<const char*>(d_y);
    if (xb < yb + (size_t)R * 4 && yb < xb + (size_t)R * 4) return SPMV_ERR_INVALID_ARG;
  }
  DeviceGuard dg;
  SPMV_TRY(dg.set(h->device));
  SPMV_TRY(check_device_ptr(d_y, h->device));
  SPMV_TRY(check_device_ptr(d_x, h->device));
  spmv::CgState* host = pinned_cg_buffer();
  if (!host) return SPMV_ERR_ALLOC;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  h->lastStream = s;
  // work: g, two d buffers, q (each padded to 64 floats), the per-block
  // partial sums and the state
  const long long pitch = (R + 63) / 64 * 64;
  const size_t nPart = spmv::cg_partials_floats();
  std::vector<Buf> tmp;
  void* work = nullptr;
  int st = h->alloc(sizeof(float) * (4 * (size_t)pitch + nPart) + sizeof(spmv::CgState), s,
                    &work, tmp);
  auto done = [&](int code) {
    h->release(tmp, s);
    return code;
  };
  if (st != SPMV_OK) return done(st);
  float* g = static_cast<float*>(work);
  float* dBuf[2] = {g + pitch, g + 2 * pitch};
  float* q = g + 3 * pitch;
  float* partials = g + 4 * pitch;
  auto* state = reinterpret_cast<spmv::CgState*>(partials + nPart);
  const bool fusedEll = format == SPMV_ELL;
  st = record(cudaMemsetAsync(state, 0, sizeof(spmv::CgState), s));
  // both d buffers start at 0: with beta = 0 the first direction is -g
  if (st == SPMV_OK)
    st = record(cudaMemsetAsync(dBuf[0], 0, sizeof(float) * 2 * (size_t)pitch, s));
  // g_0 = A·X_0 + Y: the SpMV-and-accumulate itself
  if (st == SPMV_OK)
    st = record(cudaMemcpyAsync(g, d_y, sizeof(float) * (size_t)R, cudaMemcpyDeviceToDevice, s));
  if (st == SPMV_OK) st = run_format(h, format, d_x, g, s);
  if (st == SPMV_OK) st = record(spmv::launch_cg_start((int)R, g, d_y, tol, partials, state, s));
  auto read_state = [&]() {
    int e = record(cudaMemcpyAsync(host, state, sizeof(spmv::CgState), cudaMemcpyDeviceToHost, s));
    if (e == SPMV_OK) e = record(cudaStreamSynchronize(s));
    return e;
  };
  // Iterations are enqueued in batches; the device stops itself at
  // convergence, the host reads the state between batches (after 1, 2, 4, ...,
  // 64 iterations, then every 64) so as not to enqueue far past the stop.
  int enq = 0, nextCheck = 1;
  if (st == SPMV_OK && maxIter > 0) {
    st = read_state();
    if (st == SPMV_OK && host->status != spmv::kCgRunning) nextCheck = -1;
  }
  while (st == SPMV_OK && nextCheck > 0 && enq < maxIter) {
    float* d = dBuf[(enq + 1) & 1];
    if (fusedEll) {
      // d = -g + beta d_old, q = A d, d'q in one kernel (d_old: the other buffer)
      st = record(spmv::launch_cg_ell_q((int)R, h->ellK, h->ellCol, cval<float>(h->ellVal), g,
                                        dBuf[enq & 1],
                                        d, q, partials, state, s));
    } else {
      d = dBuf[0];
      st = record(spmv::launch_cg_direction((int)R, g, d, state, s));
      if (st == SPMV_OK) st = record(cudaMemsetAsync(q, 0, sizeof(float) * (size_t)R, s));
      if (st == SPMV_OK) st = run_format(h, format, d, q, s);
      if (st == SPMV_OK) st = record(spmv::launch_cg_dot((int)R, d, q, partials, state, s));
    }
    if (st == SPMV_OK)
      st = record(spmv::launch_cg_update((int)R, d_x, g, d, q, partials, state, s));
    ++enq;
    if (st == SPMV_OK && (enq == nextCheck || enq == maxIter)) {
      st = read_state();
      if (st == SPMV_OK && host->status != spmv::kCgRunning) break;
      nextCheck = nextCheck < 64 ? nextCheck * 2 : nextCheck + 64;
    }
  }
  if (st == SPMV_OK) st = read_state();
  if (st != SPMV_OK) return done(st);
  info->iterations = host->iter;
  info->status = host->status == spmv::kCgRunning ? spmv::kCgMaxIter : host->status;
  info->residual_norm = host->gnorm;
  info->y_norm = host->ynorm;
  return done(SPMV_OK);
}

int spmv_get_stats(spmv_handle h, spmv_stats* out) {
  SPMV_TRY(check_handle(h));
  if (!out) return SPMV_ERR_INVALID_ARG;
  *out = h->stats;
  return SPMV_OK;
}

int spmv_export(spmv_handle h, spmv_format format, spmv_arrays* out) {
  SPMV_TRY(check_handle(h));
  if (!out) return SPMV_ERR_INVALID_ARG;
  std::memset(out, 0, sizeof(*out));
  out->format = format;
  out->num_rows = h->R;
  out->num_cols = h->C;
  out->nnz = h->Z;
  out->value_bytes = h->f64 ? (int32_t)sizeof(double) : (int32_t)sizeof(float);
  // value arrays go to the field of the handle's value type
  auto setv = [&](const void* v) {
    if (h->f64)
      out->value_f64 = static_cast<const double*>(v);
    else
      out->value = static_cast<const float*>(v);
  };
  auto setcv = [&](const void* v) {
    if (h->f64)
      out->coo_value_f64 = static_cast<const double*>(v);
    else
      out->coo_value = static_cast<const float*>(v);
  };
  switch (format) {
    case SPMV_CSR:
      out->row_ptrs = h->rowPtrs;
      out->col_idx = h->colIdx;
      setv(h->value);
      return SPMV_OK;
    case SPMV_COO:
      if (!h->hasCoo) return SPMV_ERR_NOT_CONVERTED;
      out->row_idx = h->cooRow;
      out->col_idx = h->colIdx;
      setv(h->value);
      out->coo_nnz = h->Z;
      return SPMV_OK;
    case SPMV_ELL:
      if (!h->hasEll) return SPMV_ERR_NOT_CONVERTED;
      out->width = h->ellK;
      out->ell_slots = (int64_t)h->R * h->ellK;
      out->col_idx = h->ellCol;
      setv(h->ellVal);
      out->nnz_per_row = h->ellNnz;
      return SPMV_OK;
    case SPMV_HYB:
      if (!h->hasHyb) return SPMV_ERR_NOT_CONVERTED;
      out->width = h->hybK;
      out->ell_slots = (int64_t)h->R * h->hybK;
      out->col_idx = h->hybCol;
      setv(h->hybVal);
      out->nnz_per_row = h->hybNnz;
      out->coo_nnz = h->hybCooN;
      out->row_idx = h->hybCooRow;
      out->coo_col_idx = h->hybCooCol;
      setcv(h->hybCooVal);
      return SPMV_OK;
    case SPMV_JDS:
      if (!h->hasJds) return SPMV_ERR_NOT_CONVERTED;
      out->width = h->jdsMaxLen;
      out->col_idx = h->jdsCol;
      setv(h->jdsVal);
      out->perm = h->jdsPerm;
      out->iter_ptr = h->jdsIterPtr;
      return SPMV_OK;
    case SPMV_SELL:
      if (!h->hasSell) return SPMV_ERR_NOT_CONVERTED;
      out->width = h->sellW0;
      out->ell_slots = h->sellSlots;
      out->col_idx = h->sellCol;
      setv(h->sellVal);
      out->perm = h->sellPerm;
      out->sec_ptr = h->sellSecPtr;
      out->section_rows = h->sellS;
      return SPMV_OK;
    case SPMV_XBLOCK:
      if (!h->hasXb) return SPMV_ERR_NOT_CONVERTED;
      if (h->xbSlots < 0) {  // the slot count lives on the device
        int n = 0;
        DeviceGuard g;
        SPMV_TRY(g.set(h->device));
        SPMV_TRY(record(cudaMemcpyAsync(&n, h->xbChunkPtr + h->xbNch, sizeof(int),
                                        cudaMemcpyDeviceToHost, h->lastStream)));
        SPMV_TRY(record(cudaStreamSynchronize(h->lastStream)));
        h->xbSlots = n;
      }
      out->ell_slots = h->xbSlots;
      out->row_idx = h->xbRow;
      setv(h->xbVal);
      out->chunk_ptr = h->xbChunkPtr;
      out->col16 = h->xbCol;
      out->chunk_cols = h->xbB;
      out->num_chunks = h->xbNch;
      return SPMV_OK;
    default:
      return SPMV_ERR_INVALID_ARG;
  }
}

int spmv_destroy(spmv_handle h) {
  if (!h) return SPMV_OK;
  DeviceGuard g;
  int st = g.set(h->device);
  cudaStream_t s = h->lastStream;
  h->release(h->csrBufs, s);
  h->release(h->cooBufs, s);
  h->release(h->ellBufs, s);
  h->release(h->hybBufs, s);
  h->release(h->jdsBufs, s);
  h->release(h->sellBufs, s);
  h->release(h->xbBufs, s);
  delete h;
  return st;
}

const char* spmv_status_string(int status) {
  switch (status) {
    case SPMV_OK: return "ok";
    case SPMV_ERR_INVALID_ARG: return "invalid argument";
    case SPMV_ERR_BAD_ROWPTRS: return "rowPtrs must start at 0, never decrease and end at nnz";
    case SPMV_ERR_COL_OUT_OF_RANGE: return "a column index is negative or not below numCols";
    case SPMV_ERR_TOO_LARGE: return "ELL slot count exceeds int32 or the padding budget";
    case SPMV_ERR_NOT_CONVERTED: return "format not converted";
    case SPMV_ERR_CUDA: return "CUDA runtime error";
    case SPMV_ERR_ALLOC: return "device allocation failed or exceeded the memory limit";
    case SPMV_ERR_TIMEOUT: return "device wait timed out";
    default: return "unknown status";
  }
}

int spmv_last_cuda_error(void) { return g_lastCudaError; }

uint64_t spmv_launch_count(void) { return g_launches.load(); }

int spmv_set_memory_limit(int64_t bytes) {
  g_memLimit.store(bytes < 0 ? -1 : bytes);
  return SPMV_OK;
}

int spmv_version(void) { return 1 * 10000 + 0 * 100 + 0; }

}  // extern "C"
