// fln_tp.cu -- the TPSP region across tensor-parallel ranks: a row-parallel
// projection whose AllReduce boundary becomes ReduceScatter -> residual add +
// RMSNorm on a token shard -> AllGather, pipelined in microchunks.
//
// What it computes follows the vLLM "TPSP Design" page: section 1
// "Motivation" (each rank holds a K-shard of the projection's input and
// weight and computes a partial y over all tokens; ReduceScatter over tokens
// leaves each rank the summed y of about T / P tokens with the complete
// hidden dimension; it adds that to its token-sharded residual and normalises
// those rows; AllGather returns the full [T, H] normalised tensor to every
// rank for the next projection), section 3 "Microchunk pipeline" (per chunk
// GEMM -> RS -> add/norm -> AG; later GEMMs overlap earlier chunks'
// communication and norm on a second stream; three reusable slots guarded by
// readiness / completion events; uneven token partitions padded, only valid
// rows update residuals and outputs) and section 4 "Constraints" (BF16,
// microchunks of at most 4096 tokens per rank, a shared workspace that
// assumes sequential calls).
//
// Token partition (the reading taken where the page leaves it open): the T
// tokens are split into P shards of S = ceil(T / P) rows, rank p owning tokens
// [p S, min((p + 1) S, T)) -- the padded uneven partition; its residual is
// that shard ([S, H], rows past T never touched).  A microchunk of c tokens
// per rank is chunk i of every shard at once: rank p's rows [i c, i c + n_i)
// of its shard, n_i = min(c, S - i c).  The chunk's GEMM computes the partial
// y of all P blocks into a rank-major slot [P, n_i, H] (fp32), exactly the
// ReduceScatter input layout, so the collective needs no repacking; the
// gathered blocks are scattered back to token order, valid rows only.
//
// The collectives are NCCL's (loaded at run time from the process, e.g. the
// copy PyTorch loaded, so the library itself has no link-time dependency).
// The partial y stays fp32 through the ReduceScatter (y is never rounded
// before the residual add, as on one GPU); the gathered output is bf16.
#include <dlfcn.h>

#include <algorithm>
#include <cstdint>
#include <cstdlib>
#include <cstring>

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "fln_internal.h"
#include "libfusedln.h"

using namespace fln;

namespace {

constexpr int kMaxChunk = 4096;        // per-rank microchunk cap ("TPSP Design", section 4)
constexpr int kDefaultChunk = 1024;    // microchunk when the caller passes 0
constexpr int kTile = 256;             // GEMM tile width on H

// ------------------------------------------------------------------ NCCL, resolved at run time
// The few entry points used, with the library's published C signatures
// (enumerations passed as int, the communicator as an opaque pointer, the
// unique id as its 128-byte struct).
typedef int nccl_result;
struct NcclId {
  char internal[128];
};
typedef struct NcclCommOpaque* nccl_comm;
constexpr nccl_result kNcclSuccess = 0;
constexpr int kNcclSum = 0;
constexpr int kNcclFloat32 = 7;
constexpr int kNcclBfloat16 = 9;

struct NcclApi {
  nccl_result (*get_unique_id)(NcclId*) = nullptr;
  nccl_result (*comm_init_rank)(nccl_comm*, int, NcclId, int) = nullptr;
  nccl_result (*comm_init_all)(nccl_comm*, int, const int*) = nullptr;
  nccl_result (*comm_destroy)(nccl_comm) = nullptr;
  nccl_result (*reduce_scatter)(const void*, void*, size_t, int, int, nccl_comm, cudaStream_t) = nullptr;
  nccl_result (*all_gather)(const void*, void*, size_t, int, nccl_comm, cudaStream_t) = nullptr;
  const char* (*error_string)(nccl_result) = nullptr;
  bool loaded = false;
};

NcclApi g_nccl;

// Finds NCCL: a copy already in the process first (PyTorch loads one), then
// the FLN_NCCL_LIBRARY path, then the loader's search path.
int load_nccl() {
  if (g_nccl.loaded) return FLN_OK;
  const char* env = std::getenv("FLN_NCCL_LIBRARY");
  const char* names[] = {env, "libnccl.so.2", "libnccl.so"};
  void* h = nullptr;
  for (const char* n : names)
    if (n && !h) h = dlopen(n, RTLD_NOW | RTLD_NOLOAD);
  for (const char* n : names)
    if (n && !h) h = dlopen(n, RTLD_NOW | RTLD_GLOBAL);
  if (!h) return api_fail(FLN_ERR_COMM, "NCCL is not available (libnccl.so.2 not found; set FLN_NCCL_LIBRARY)");
  NcclApi a;
  a.get_unique_id = reinterpret_cast<decltype(a.get_unique_id)>(dlsym(h, "ncclGetUniqueId"));
  a.comm_init_rank = reinterpret_cast<decltype(a.comm_init_rank)>(dlsym(h, "ncclCommInitRank"));
  a.comm_init_all = reinterpret_cast<decltype(a.comm_init_all)>(dlsym(h, "ncclCommInitAll"));
  a.comm_destroy = reinterpret_cast<decltype(a.comm_destroy)>(dlsym(h, "ncclCommDestroy"));
  a.reduce_scatter = reinterpret_cast<decltype(a.reduce_scatter)>(dlsym(h, "ncclReduceScatter"));
  a.all_gather = reinterpret_cast<decltype(a.all_gather)>(dlsym(h, "ncclAllGather"));
  a.error_string = reinterpret_cast<decltype(a.error_string)>(dlsym(h, "ncclGetErrorString"));
  if (!a.get_unique_id || !a.comm_init_rank || !a.comm_init_all || !a.comm_destroy || !a.reduce_scatter ||
      !a.all_gather || !a.error_string)
    return api_fail(FLN_ERR_COMM, "the NCCL library found lacks an entry point the TP region needs");
  a.loaded = true;
  g_nccl = a;
  return FLN_OK;
}

int nccl_fail(nccl_result r, const char* what) {
  return api_fail(FLN_ERR_COMM, "%s: NCCL error %d (%s)", what, r, g_nccl.error_string ? g_nccl.error_string(r) : "");
}

#define TP_CUDA(call, what)                             \
  do {                                                  \
    cudaError_t e_ = (call);                            \
    if (e_ != cudaSuccess) return api_cuda_fail(e_, what); \
  } while (0)

#define TP_NCCL(call, what)                         \
  do {                                              \
    nccl_result r_ = (call);                        \
    if (r_ != kNcclSuccess) return nccl_fail(r_, what); \
  } while (0)

// ------------------------------------------------------------------ partition
struct Layout {
  int S;       // shard rows per rank, ceil(T / P)
  int c;       // microchunk rows per rank
  int chunks;  // ceil(S / c)
};

int layout_of(int T, int P, int chunk_arg, Layout* L) {
  if (T < 0 || P < 1) return api_fail(FLN_ERR_INVALID_ARG, "T=%d, nranks=%d", T, P);
  if (chunk_arg < 0 || chunk_arg > kMaxChunk)
    return api_fail(FLN_ERR_INVALID_ARG, "microchunk_tokens=%d outside 0..%d", chunk_arg, kMaxChunk);
  L->S = T == 0 ? 0 : (T + P - 1) / P;
  L->c = std::max(1, std::min(chunk_arg > 0 ? chunk_arg : kDefaultChunk, std::max(L->S, 1)));
  L->chunks = L->S == 0 ? 0 : (L->S + L->c - 1) / L->c;
  return FLN_OK;
}

// chunk i of rank q: first token, block rows (the same on every rank), valid rows
void chunk_of(int T, const Layout& L, int i, int q, int* token0, int* rows, int* valid) {
  const int r0 = i * L.c;
  const int n = std::min(L.c, L.S - r0);
  const long long t0 = static_cast<long long>(q) * L.S + r0;
  *token0 = static_cast<int>(std::min<long long>(t0, T));
  *rows = n;
  *valid = static_cast<int>(std::max<long long>(0, std::min<long long>(n, T - t0)));
}

// ------------------------------------------------------------------ gathered rows back to token order
// gath [P, n, H] (rank-major blocks of the chunk) -> out rows q S + r0 + j for
// j < n and q S + r0 + j < T; 16 bytes a thread, grid-stride.
__global__ void tp_scatter_rows_kernel(const uint4* __restrict__ gath, uint4* __restrict__ out, int P, int n,
                                       int H8, int S, int r0, int T) {
  const long long per_block = static_cast<long long>(n) * H8;
  const long long total = per_block * P;
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const int q = static_cast<int>(i / per_block);
    const long long rem = i - q * per_block;
    const int j = static_cast<int>(rem / H8);
    const int c = static_cast<int>(rem - static_cast<long long>(j) * H8);
    const long long tok = static_cast<long long>(q) * S + r0 + j;
    if (tok < T) out[tok * H8 + c] = gath[i];
  }
}

}  // namespace

// One rank's handle: the NCCL communicator, the second stream, three slots of
// each pipeline buffer and their events.  Sequential use, like the workspace.
struct fln_tp_comm {
  int nranks = 0, rank = 0, device = -1, sms = 0;
  nccl_comm comm = nullptr;
  cudaStream_t stream_b = nullptr;
  cudaEvent_t ev_ready[3] = {}, ev_free[3] = {}, ev_join = nullptr;
  float* slot[3] = {};             // [P, n, H] partial y of a chunk, rank-major blocks (fp32)
  float* red[3] = {};              // [n, H] this rank's summed y of the chunk (fp32)
  __nv_bfloat16* send[3] = {};     // [n, H] this rank's normalised rows of the chunk
  __nv_bfloat16* gath[3] = {};     // [P, n, H] every rank's normalised rows of the chunk
  size_t rows_cap = 0, h_cap = 0;  // buffers hold chunks of rows_cap rows of h_cap columns
  bool prepared = false;
};

namespace {

void free_buffers(fln_tp_comm* c) {
  for (int i = 0; i < 3; ++i) {
    cudaFree(c->slot[i]);
    cudaFree(c->red[i]);
    cudaFree(c->send[i]);
    cudaFree(c->gath[i]);
    c->slot[i] = c->red[i] = nullptr;
    c->send[i] = c->gath[i] = nullptr;
  }
  c->rows_cap = c->h_cap = 0;
}

int ensure_buffers(fln_tp_comm* c, int rows, int H) {
  if (static_cast<size_t>(rows) <= c->rows_cap && static_cast<size_t>(H) <= c->h_cap) return FLN_OK;
  TP_CUDA(cudaDeviceSynchronize(), "cudaDeviceSynchronize before TP buffer growth");
  free_buffers(c);
  const size_t n = static_cast<size_t>(rows) * H, P = static_cast<size_t>(c->nranks);
  for (int i = 0; i < 3; ++i) {
    TP_CUDA(cudaMalloc(&c->slot[i], P * n * sizeof(float)), "cudaMalloc(TP slot)");
    TP_CUDA(cudaMalloc(&c->red[i], n * sizeof(float)), "cudaMalloc(TP reduced rows)");
    TP_CUDA(cudaMalloc(&c->send[i], n * sizeof(__nv_bfloat16)), "cudaMalloc(TP normalised rows)");
    TP_CUDA(cudaMalloc(&c->gath[i], P * n * sizeof(__nv_bfloat16)), "cudaMalloc(TP gathered rows)");
  }
  c->rows_cap = rows;
  c->h_cap = H;
  return FLN_OK;
}

int make_comm(int nranks, int rank, const void* id, fln_tp_comm** out) {
  api_lock();
  int rc = load_nccl();
  api_unlock();
  if (rc) return rc;
  fln_tp_comm* c = new fln_tp_comm();
  c->nranks = nranks;
  c->rank = rank;
  cudaError_t e = cudaGetDevice(&c->device);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&c->sms, cudaDevAttrMultiProcessorCount, c->device);
  int lo = 0, hi = 0;
  if (e == cudaSuccess) e = cudaDeviceGetStreamPriorityRange(&lo, &hi);
  if (e == cudaSuccess) e = cudaStreamCreateWithPriority(&c->stream_b, cudaStreamNonBlocking, hi);
  for (int i = 0; i < 3 && e == cudaSuccess; ++i) {
    e = cudaEventCreateWithFlags(&c->ev_ready[i], cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&c->ev_free[i], cudaEventDisableTiming);
  }
  if (e == cudaSuccess) e = cudaEventCreateWithFlags(&c->ev_join, cudaEventDisableTiming);
  if (e != cudaSuccess) {
    delete c;
    return api_cuda_fail(e, "TP communicator set-up");
  }
  nccl_result r;
  if (!id) {
    // one rank in this process: no rendezvous needed
    r = g_nccl.comm_init_all(&c->comm, 1, &c->device);
  } else {
    NcclId uid;
    std::memcpy(&uid, id, sizeof uid);
    r = g_nccl.comm_init_rank(&c->comm, nranks, uid, rank);
  }
  cudaSetDevice(c->device);  // the initialisation may have switched devices
  if (r != kNcclSuccess) {
    delete c;
    return nccl_fail(r, "NCCL communicator initialisation");
  }
  *out = c;
  return FLN_OK;
}

}  // namespace

extern "C" {

int fln_tp_unique_id(void* id) {
  api_lock();
  int rc = id ? load_nccl() : api_fail(FLN_ERR_INVALID_ARG, "id is NULL");
  if (!rc) {
    NcclId uid;
    nccl_result r = g_nccl.get_unique_id(&uid);
    if (r != kNcclSuccess) {
      rc = nccl_fail(r, "ncclGetUniqueId");
    } else {
      std::memcpy(id, &uid, sizeof uid);
    }
  }
  api_unlock();
  return rc;
}

int fln_tp_comm_init(int nranks, int rank, const void* id, fln_tp_comm** comm) {
  api_lock();
  int rc = FLN_OK;
  if (!comm) rc = api_fail(FLN_ERR_INVALID_ARG, "comm is NULL");
  else if (nranks < 1 || rank < 0 || rank >= nranks)
    rc = api_fail(FLN_ERR_INVALID_ARG, "rank %d of %d ranks", rank, nranks);
  else if (!id && nranks != 1)
    rc = api_fail(FLN_ERR_INVALID_ARG, "a unique id is needed for %d ranks", nranks);
  api_unlock();
  if (rc) return rc;
  // not under the library lock: the initialisation waits for the other ranks
  return make_comm(nranks, rank, id, comm);
}

int fln_tp_comm_destroy(fln_tp_comm* c) {
  if (!c) return FLN_OK;
  api_lock();
  int cur = 0;
  cudaGetDevice(&cur);
  cudaSetDevice(c->device);
  cudaDeviceSynchronize();
  free_buffers(c);
  for (int i = 0; i < 3; ++i) {
    cudaEventDestroy(c->ev_ready[i]);
    cudaEventDestroy(c->ev_free[i]);
  }
  cudaEventDestroy(c->ev_join);
  cudaStreamDestroy(c->stream_b);
  nccl_result r = c->comm ? g_nccl.comm_destroy(c->comm) : kNcclSuccess;
  cudaSetDevice(cur);
  delete c;
  int rc = r == kNcclSuccess ? FLN_OK : nccl_fail(r, "ncclCommDestroy");
  api_unlock();
  return rc;
}

int fln_tp_layout(int T, int nranks, int microchunk_tokens, int* shard_rows, int* chunk_tokens, int* num_chunks) {
  Layout L;
  int rc = layout_of(T, nranks, microchunk_tokens, &L);
  if (rc) return rc;
  if (shard_rows) *shard_rows = L.S;
  if (chunk_tokens) *chunk_tokens = L.c;
  if (num_chunks) *num_chunks = L.chunks;
  return FLN_OK;
}

int fln_tp_chunk_rows(int T, int nranks, int microchunk_tokens, int chunk, int rank, int* token0, int* rows,
                      int* valid) {
  Layout L;
  int rc = layout_of(T, nranks, microchunk_tokens, &L);
  if (rc) return rc;
  if (chunk < 0 || chunk >= L.chunks || rank < 0 || rank >= nranks)
    return api_fail(FLN_ERR_INVALID_ARG, "chunk %d of %d, rank %d of %d", chunk, L.chunks, rank, nranks);
  int a, b, v;
  chunk_of(T, L, chunk, rank, &a, &b, &v);
  if (token0) *token0 = a;
  if (rows) *rows = b;
  if (valid) *valid = v;
  return FLN_OK;
}

int fused_proj_rs_add_rmsnorm_ag(const fln_bf16* x, const fln_bf16* W, fln_bf16* residual_shard,
                                 const float* gamma, float eps, int norm_kind, int T, int K, int H,
                                 int microchunk_tokens, fln_bf16* out, fln_tp_comm* comm, fln_stream_t stream) {
  api_lock();
  struct Unlock {
    ~Unlock() { api_unlock(); }
  } unlock_at_return;
  if (!comm) return api_fail(FLN_ERR_INVALID_ARG, "comm is NULL");
  int rc = api_check_common(eps, norm_kind, T, H);
  if (rc) return rc;
  if (K < 8 || (K & 7)) return api_fail(FLN_ERR_INVALID_ARG, "K=%d must be a positive multiple of 8", K);
  Layout L;
  if ((rc = layout_of(T, comm->nranks, microchunk_tokens, &L))) return rc;
  if (T == 0) return FLN_OK;
  int dev = 0;
  TP_CUDA(cudaGetDevice(&dev), "cudaGetDevice");
  if (dev != comm->device)
    return api_fail(FLN_ERR_INVALID_ARG, "the communicator belongs to device %d, the current device is %d",
                    comm->device, dev);
  if ((rc = api_check_ptr("x", x)) || (rc = api_check_ptr("W", W)) ||
      (rc = api_check_ptr("residual_shard", residual_shard)) || (rc = api_check_ptr("gamma", gamma)) ||
      (rc = api_check_ptr("out", out)))
    return rc;
  const size_t bx = size_t(T) * K * 2, bw = size_t(H) * K * 2, bs = size_t(L.S) * H * 2, bo = size_t(T) * H * 2;
  if (api_overlaps(out, bo, x, bx) || api_overlaps(out, bo, W, bw) || api_overlaps(out, bo, residual_shard, bs) ||
      api_overlaps(out, bo, gamma, size_t(H) * 4))
    return api_fail(FLN_ERR_INVALID_ARG, "out overlaps an input");
  if (api_overlaps(residual_shard, bs, x, bx) || api_overlaps(residual_shard, bs, W, bw) ||
      api_overlaps(residual_shard, bs, gamma, size_t(H) * 4))
    return api_fail(FLN_ERR_INVALID_ARG, "residual_shard overlaps x, W or gamma");
  if ((rc = ensure_buffers(comm, L.c, H))) return rc;
  unsigned int* err_word = nullptr;  // the device's error word (fln_device_status reads it)
  if ((rc = api_device_error_word(&err_word))) return rc;
  if (!comm->prepared) {
    TP_CUDA(gemm_prepare(kTile, EPI_STORE_F32, 0), "cudaFuncSetAttribute(max dynamic shared memory)");
    comm->prepared = true;
  }
  CUtensorMap tmA, tmB;
  if ((rc = api_make_map_bf16(&tmA, x, K, T, 128)) || (rc = api_make_map_bf16(&tmB, W, K, H, kTile))) return rc;
  const cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  const int P = comm->nranks;
  const int nt = (H + kTile - 1) / kTile;
  for (int i = 0; i < L.chunks; ++i) {
    const int s = i % 3;
    int tok0, n, valid;
    chunk_of(T, L, i, comm->rank, &tok0, &n, &valid);
    const int r0 = i * L.c;  // first shard row of the chunk (every rank)
    // the slot is free once the second stream is done with its previous chunk
    if (i >= 3) TP_CUDA(cudaStreamWaitEvent(cs, comm->ev_free[s], 0), "cudaStreamWaitEvent(slot free)");
    // partial y of every rank's rows of this chunk, rank-major blocks
    GemmParams p{};
    p.N = H;
    p.K = K;
    p.a_row0 = r0;
    p.blk_m_tiles = (n + 127) / 128;
    p.blk_rows = n;
    p.blk_stride = L.S;
    p.M = P * n;
    p.num_m_tiles = P * p.blk_m_tiles;
    p.num_n_tiles = nt;
    p.num_k_blocks = (K + 63) / 64;
    p.ld = H;
    p.yout = comm->slot[s];
    p.err = err_word;
    const int tiles = p.num_m_tiles * nt;
    const int G = std::max(1, std::min(comm->sms, tiles));
    TP_CUDA(launch_gemm(EPI_STORE_F32, kTile, 0, tmA, tmB, p, G, cs), "TP slot GEMM launch");
    api_count_launch();
    TP_CUDA(cudaEventRecord(comm->ev_ready[s], cs), "cudaEventRecord(slot ready)");
    TP_CUDA(cudaStreamWaitEvent(comm->stream_b, comm->ev_ready[s], 0), "cudaStreamWaitEvent(slot ready)");
    // ReduceScatter over tokens: block q of every rank's slot, summed, lands on rank q
    TP_NCCL(g_nccl.reduce_scatter(comm->slot[s], comm->red[s], static_cast<size_t>(n) * H, kNcclFloat32, kNcclSum,
                                  comm->comm, comm->stream_b),
            "ncclReduceScatter");
    if (valid > 0) {
      // residual add + norm of this rank's valid rows; normalised rows to the send buffer
      NormParams np{};
      np.y_f32 = comm->red[s];
      np.residual = reinterpret_cast<__nv_bfloat16*>(residual_shard);
      np.out = comm->send[s];
      np.out_local = 1;
      np.gamma = gamma;
      np.eps = eps;
      np.norm_kind = norm_kind;
      np.T = valid;
      np.row0 = r0;
      np.H = H;
      TP_CUDA(launch_add_rmsnorm(NORM_SRC_F32, np, 0, comm->stream_b), "TP add+norm launch");
      api_count_launch();
    }
    // AllGather of every rank's normalised rows (padding rows travel but are never used)
    TP_NCCL(g_nccl.all_gather(comm->send[s], comm->gath[s], static_cast<size_t>(n) * H, kNcclBfloat16, comm->comm,
                              comm->stream_b),
            "ncclAllGather");
    const long long vec = static_cast<long long>(P) * n * (H / 8);
    const int grid = static_cast<int>(std::min<long long>((vec + 255) / 256, 4LL * comm->sms));
    tp_scatter_rows_kernel<<<grid, 256, 0, comm->stream_b>>>(reinterpret_cast<const uint4*>(comm->gath[s]),
                                                             reinterpret_cast<uint4*>(out), P, n, H / 8, L.S, r0, T);
    TP_CUDA(cudaGetLastError(), "TP row scatter launch");
    api_count_launch();
    TP_CUDA(cudaEventRecord(comm->ev_free[s], comm->stream_b), "cudaEventRecord(slot free)");
  }
  TP_CUDA(cudaEventRecord(comm->ev_join, comm->stream_b), "cudaEventRecord(join)");
  TP_CUDA(cudaStreamWaitEvent(cs, comm->ev_join, 0), "cudaStreamWaitEvent(join)");
  return FLN_OK;
}

}  // extern "C"
