// The Ulysses block across real GPUs: one process (rank) per GPU, the two all-to-alls as
// NCCL exchanges between them ("Snowflake's Ulysses trick trains transformers on
// million-token contexts across GPUs", para 2: local QKV projection, an all-to-all that
// leaves each GPU the full sequence for a subset of heads, attention per head group, and an
// all-to-all back; para 3: two all-to-alls per layer, O(hidden x seq_len / P) per rank).
//
// A rank holds n = S/P tokens.  Its send and receive buffers are block-major: block p,
// one contiguous run of n * (heads/P) * D elements, goes to (comes from) rank p.  With
// that layout the received q, k, v blocks are, in token order, exactly the head layout the
// attention kernels read ([S][heads/P][D]), and the attention's o is, as it stands, the send
// buffer of the way back.  So the data plane needs only a pack before the first exchange
// (the permute kernel run over the shard, RoPE at the tokens' global positions) and an
// unpack after the second; no kernel touches another GPU's memory.
//
// The exchange is one NCCL group of P sends and P receives per buffer.  NCCL is loaded at
// run time (dlopen of libnccl.so.2), so the library links and runs without it wherever no
// exchange is asked for.
#include <dlfcn.h>

#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <type_traits>

#include "uly_internal.h"

namespace uly {
namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

uly_status err(uly_status s, const char* fmt, ...) __attribute__((format(printf, 2, 3)));
uly_status err(uly_status s, const char* fmt, ...) {
  char msg[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(msg, sizeof(msg), fmt, ap);
  va_end(ap);
  return set_error(s, msg);
}

uly_status need_rank_plan(uly_plan plan, const char* what) {
  if (!plan) return set_error(ULY_ERR_INVALID_ARG, "plan is NULL");
  if (plan->p.rank < 0)
    return err(ULY_ERR_INVALID_ARG, "%s needs a rank plan (ulysses_plan_rank)", what);
  return ULY_OK;
}

// ---------------------------------------------------------------------------- NCCL
// The few NCCL entry points the exchange uses, resolved from libnccl.so.2.  The id is a
// 128-byte struct passed by value; results and data types are C enums (ncclInt8 = 0).
struct NcclId {
  char internal[128];
};
struct Nccl {
  void* handle = nullptr;
  int (*get_unique_id)(NcclId*) = nullptr;
  int (*comm_init_rank)(void**, int, NcclId, int) = nullptr;
  int (*comm_destroy)(void*) = nullptr;
  int (*comm_count)(const void*, int*) = nullptr;
  int (*comm_user_rank)(const void*, int*) = nullptr;
  int (*send)(const void*, size_t, int, int, void*, cudaStream_t) = nullptr;
  int (*recv)(void*, size_t, int, int, void*, cudaStream_t) = nullptr;
  int (*group_start)() = nullptr;
  int (*group_end)() = nullptr;
  const char* (*error_string)(int) = nullptr;
  char why[256] = "";
};
constexpr int kNcclInt8 = 0;

const Nccl& nccl() {
  static Nccl n;
  static std::once_flag once;
  std::call_once(once, [] {
    const char* env = getenv("ULY_NCCL_LIBRARY");
    const char* names[] = {env, "libnccl.so.2", "libnccl.so"};
    for (const char* name : names) {
      if (!name) continue;
      n.handle = dlopen(name, RTLD_NOW | RTLD_LOCAL);
      if (n.handle) break;
    }
    if (!n.handle) {
      snprintf(n.why, sizeof(n.why), "libnccl.so.2 could not be loaded (%s)", dlerror());
      return;
    }
    auto sym = [&](const char* name, auto& fn) {
      fn = reinterpret_cast<std::remove_reference_t<decltype(fn)>>(dlsym(n.handle, name));
      if (!fn && !n.why[0]) snprintf(n.why, sizeof(n.why), "NCCL lacks %s", name);
    };
    sym("ncclGetUniqueId", n.get_unique_id);
    sym("ncclCommInitRank", n.comm_init_rank);
    sym("ncclCommDestroy", n.comm_destroy);
    sym("ncclCommCount", n.comm_count);
    sym("ncclCommUserRank", n.comm_user_rank);
    sym("ncclSend", n.send);
    sym("ncclRecv", n.recv);
    sym("ncclGroupStart", n.group_start);
    sym("ncclGroupEnd", n.group_end);
    sym("ncclGetErrorString", n.error_string);
    if (n.why[0]) {
      dlclose(n.handle);
      n.handle = nullptr;
    }
  });
  return n;
}

uly_status nccl_ready() {
  const Nccl& n = nccl();
  if (!n.handle) return err(ULY_ERR_UNSUPPORTED, "NCCL is not available: %s", n.why);
  return ULY_OK;
}

uly_status nccl_fail(int r, const char* what) {
  return err(ULY_ERR_CUDA, "%s: NCCL error %d (%s)", what, r, nccl().error_string(r));
}

}  // namespace
}  // namespace uly

using uly::Plan;

extern "C" {

uly_status ulysses_a2a_table(const uly_config* cfg, int32_t rank, int32_t to_head,
                             int32_t n_heads, uly_a2a_block* blocks) {
  if (!cfg || !blocks) return uly::set_error(ULY_ERR_INVALID_ARG, "NULL argument");
  if (cfg->P < 1 || rank < 0 || rank >= cfg->P)
    return uly::err(ULY_ERR_INVALID_ARG, "rank %d outside [0, P = %d)", rank, cfg->P);
  if (n_heads != cfg->n_q_heads && n_heads != cfg->n_kv_heads)
    return uly::err(ULY_ERR_INVALID_ARG, "n_heads must be n_q_heads or n_kv_heads (got %d)",
                    n_heads);
  uint64_t v1 = 0, v2 = 0;   // validates the rest of the config
  uly_status s = ulysses_a2a_volume(cfg, &v1, &v2);
  if (s != ULY_OK) return s;
  const int P = cfg->P;
  const int64_t n = cfg->seq_len / P;
  const int hp = n_heads / P;
  const uint64_t count = (uint64_t)n * hp * cfg->head_dim;
  for (int p = 0; p < P; ++p) {
    uly_a2a_block& b = blocks[p];
    memset(&b, 0, sizeof(b));
    b.peer = p;
    b.n_tokens = (int32_t)n;
    b.n_heads = hp;
    if (to_head) {   // send: my tokens, p's heads; receive: p's tokens, my heads
      b.send_token_begin = (int64_t)rank * n;
      b.send_head_begin = p * hp;
      b.recv_token_begin = (int64_t)p * n;
      b.recv_head_begin = rank * hp;
    } else {         // send: p's tokens, my heads; receive: my tokens, p's heads
      b.send_token_begin = (int64_t)p * n;
      b.send_head_begin = rank * hp;
      b.recv_token_begin = (int64_t)rank * n;
      b.recv_head_begin = p * hp;
    }
    b.send_offset = (uint64_t)p * count;
    b.recv_offset = (uint64_t)p * count;
    b.count = count;
  }
  return uly::set_error(ULY_OK, "");
}

uly_status ulysses_a2a_pack_qkv(uly_plan plan, const void* qkv_local, int in_fp32,
                                int apply_rope, void* send_q, void* send_k, void* send_v,
                                void* stream) {
  ULY_CALL_RANGE();
  uly_status s = uly::need_rank_plan(plan, "ulysses_a2a_pack_qkv");
  if (s != ULY_OK) return s;
  const Plan& v = plan->shard;
  if (v.S == 0) return uly::set_error(ULY_OK, "");
  if (!qkv_local || !send_q || !send_k || !send_v)
    return uly::set_error(ULY_ERR_INVALID_ARG, "NULL tensor pointer");
  if (!uly::aligned16(qkv_local) || !uly::aligned16(send_q) || !uly::aligned16(send_k) ||
      !uly::aligned16(send_v))
    return uly::set_error(ULY_ERR_INVALID_ARG, "tensor pointers must be 16-byte aligned");
  if (apply_rope && !(v.cfg.rope_theta > 0))
    return uly::set_error(ULY_ERR_INVALID_ARG, "apply_rope needs a plan with rope_theta > 0");
  const uint64_t elems = (uint64_t)v.S * (v.H + 2 * v.G) * v.D;
  plan->p.bytes_moved += elems * (in_fp32 ? 4 : 2) + elems * 2;
  const cudaError_t e =
      uly::launch_seq_to_head(v, qkv_local, in_fp32 != 0, apply_rope != 0, send_q, send_k,
                              send_v, reinterpret_cast<cudaStream_t>(stream),
                              (int64_t)plan->p.rank * v.S);
  if (e != cudaSuccess) return uly::err(ULY_ERR_CUDA, "a2a_pack_qkv launch: %s", cudaGetErrorString(e));
  return uly::set_error(ULY_OK, "");
}

static uly_status pack_or_unpack(uly_plan plan, const void* in, int n_heads, void* out,
                                 bool pack, void* stream) {
  uly_status s = uly::need_rank_plan(plan, pack ? "ulysses_a2a_pack_heads"
                                                : "ulysses_a2a_unpack_heads");
  if (s != ULY_OK) return s;
  const Plan& v = plan->shard;
  if (n_heads != v.H && n_heads != v.G)
    return uly::err(ULY_ERR_INVALID_ARG, "n_heads must be n_q_heads or n_kv_heads (got %d)",
                    n_heads);
  if (v.S == 0) return uly::set_error(ULY_OK, "");
  if (!in || !out) return uly::set_error(ULY_ERR_INVALID_ARG, "NULL tensor pointer");
  if (!uly::aligned16(in) || !uly::aligned16(out))
    return uly::set_error(ULY_ERR_INVALID_ARG, "tensor pointers must be 16-byte aligned");
  plan->p.bytes_moved += (uint64_t)v.S * n_heads * v.D * 2 * 2;
  const cudaError_t e = uly::launch_permute_heads(v, in, n_heads, out, pack,
                                                  reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return uly::err(ULY_ERR_CUDA, "a2a pack/unpack launch: %s", cudaGetErrorString(e));
  return uly::set_error(ULY_OK, "");
}

uly_status ulysses_a2a_pack_heads(uly_plan plan, const void* x_local, int n_heads, void* send,
                                  void* stream) {
  ULY_CALL_RANGE();
  return pack_or_unpack(plan, x_local, n_heads, send, true, stream);
}

uly_status ulysses_a2a_unpack_heads(uly_plan plan, const void* recv, int n_heads,
                                    void* x_local, void* stream) {
  ULY_CALL_RANGE();
  return pack_or_unpack(plan, recv, n_heads, x_local, false, stream);
}

uly_status ulysses_a2a_unpack_qkv(uly_plan plan, const void* recv_dq, const void* recv_dk,
                                  const void* recv_dv, int apply_rope, void* dqkv_local,
                                  void* stream) {
  ULY_CALL_RANGE();
  uly_status s = uly::need_rank_plan(plan, "ulysses_a2a_unpack_qkv");
  if (s != ULY_OK) return s;
  const Plan& v = plan->shard;
  if (v.S == 0) return uly::set_error(ULY_OK, "");
  if (!recv_dq || !recv_dk || !recv_dv || !dqkv_local)
    return uly::set_error(ULY_ERR_INVALID_ARG, "NULL tensor pointer");
  if (!uly::aligned16(recv_dq) || !uly::aligned16(recv_dk) || !uly::aligned16(recv_dv) ||
      !uly::aligned16(dqkv_local))
    return uly::set_error(ULY_ERR_INVALID_ARG, "tensor pointers must be 16-byte aligned");
  if (apply_rope && !(v.cfg.rope_theta > 0))
    return uly::set_error(ULY_ERR_INVALID_ARG, "apply_rope needs a plan with rope_theta > 0");
  plan->p.bytes_moved += (uint64_t)v.S * (v.H + 2 * v.G) * v.D * 4;
  const cudaError_t e = uly::launch_head_to_seq_qkv(
      v, recv_dq, recv_dk, recv_dv, apply_rope != 0, dqkv_local,
      reinterpret_cast<cudaStream_t>(stream), (int64_t)plan->p.rank * v.S);
  if (e != cudaSuccess) return uly::err(ULY_ERR_CUDA, "a2a_unpack_qkv launch: %s", cudaGetErrorString(e));
  return uly::set_error(ULY_OK, "");
}

uly_status ulysses_a2a_exchange(uly_plan plan, void* comm, int32_t n_buffers,
                                const void* const* send, void* const* recv,
                                const uint64_t* bytes_per_peer, void* stream) {
  ULY_CALL_RANGE();
  uly_status s = uly::need_rank_plan(plan, "ulysses_a2a_exchange");
  if (s != ULY_OK) return s;
  if (!comm || !send || !recv || !bytes_per_peer)
    return uly::set_error(ULY_ERR_INVALID_ARG, "NULL argument");
  if (n_buffers < 1 || n_buffers > 8)
    return uly::err(ULY_ERR_INVALID_ARG, "n_buffers must be 1..8 (got %d)", n_buffers);
  const int P = plan->p.P;
  for (int i = 0; i < n_buffers; ++i) {
    if (!send[i] || !recv[i]) return uly::set_error(ULY_ERR_INVALID_ARG, "NULL buffer");
    const char* sb = static_cast<const char*>(send[i]);
    const char* rb = static_cast<const char*>(recv[i]);
    const uint64_t total = bytes_per_peer[i] * (uint64_t)P;
    if (sb < rb + total && rb < sb + total)
      return uly::set_error(ULY_ERR_INVALID_ARG, "send and receive buffers overlap");
  }
  s = uly::nccl_ready();
  if (s != ULY_OK) return s;
  const uly::Nccl& n = uly::nccl();
  int count = 0, me = -1;
  int r = n.comm_count(comm, &count);
  if (r != 0) return uly::nccl_fail(r, "ncclCommCount");
  r = n.comm_user_rank(comm, &me);
  if (r != 0) return uly::nccl_fail(r, "ncclCommUserRank");
  if (count != P || me != plan->p.rank)
    return uly::err(ULY_ERR_INVALID_ARG,
                    "the communicator has %d ranks and this process is its rank %d; the plan "
                    "is rank %d of %d",
                    count, me, plan->p.rank, P);
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  r = n.group_start();
  if (r != 0) return uly::nccl_fail(r, "ncclGroupStart");
  int first_err = 0;
  for (int i = 0; i < n_buffers && !first_err; ++i) {
    const uint64_t b = bytes_per_peer[i];
    if (b == 0) continue;
    for (int p = 0; p < P && !first_err; ++p) {
      first_err = n.send(static_cast<const char*>(send[i]) + (uint64_t)p * b, b, uly::kNcclInt8,
                         p, comm, st);
      if (!first_err)
        first_err = n.recv(static_cast<char*>(recv[i]) + (uint64_t)p * b, b, uly::kNcclInt8, p,
                           comm, st);
    }
  }
  r = n.group_end();
  if (first_err) return uly::nccl_fail(first_err, "ncclSend/ncclRecv");
  if (r != 0) return uly::nccl_fail(r, "ncclGroupEnd");
  for (int i = 0; i < n_buffers; ++i)   // what this rank sends to the other ranks
    plan->p.bytes_moved += bytes_per_peer[i] * (uint64_t)(P - 1);
  return uly::set_error(ULY_OK, "");
}

uly_status ulysses_nccl_unique_id(uint8_t id[128]) {
  if (!id) return uly::set_error(ULY_ERR_INVALID_ARG, "NULL argument");
  uly_status s = uly::nccl_ready();
  if (s != ULY_OK) return s;
  uly::NcclId nid;
  const int r = uly::nccl().get_unique_id(&nid);
  if (r != 0) return uly::nccl_fail(r, "ncclGetUniqueId");
  memcpy(id, nid.internal, sizeof(nid.internal));
  return uly::set_error(ULY_OK, "");
}

uly_status ulysses_nccl_comm_init(int32_t nranks, int32_t rank, const uint8_t id[128],
                                  void** comm) {
  ULY_CALL_RANGE();
  if (!id || !comm) return uly::set_error(ULY_ERR_INVALID_ARG, "NULL argument");
  *comm = nullptr;
  if (nranks < 1 || rank < 0 || rank >= nranks)
    return uly::err(ULY_ERR_INVALID_ARG, "rank %d outside [0, nranks = %d)", rank, nranks);
  uly_status s = uly::nccl_ready();
  if (s != ULY_OK) return s;
  uly::NcclId nid;
  memcpy(nid.internal, id, sizeof(nid.internal));
  const int r = uly::nccl().comm_init_rank(comm, nranks, nid, rank);
  if (r != 0) {
    *comm = nullptr;
    return uly::nccl_fail(r, "ncclCommInitRank");
  }
  return uly::set_error(ULY_OK, "");
}

uly_status ulysses_nccl_comm_destroy(void* comm) {
  if (!comm) return uly::set_error(ULY_OK, "");
  uly_status s = uly::nccl_ready();
  if (s != ULY_OK) return s;
  const int r = uly::nccl().comm_destroy(comm);
  if (r != 0) return uly::nccl_fail(r, "ncclCommDestroy");
  return uly::set_error(ULY_OK, "");
}

}  // extern "C"
