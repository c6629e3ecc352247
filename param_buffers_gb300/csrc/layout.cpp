// Host layout engine of the flat param/grad buffers.
//
// Follows "05 · grad/param buffer: contiguous buffer data structures and read/write
// loop" (llm-infra-atlas): §3 BufferKey grouping, §4.1 reverse (backprop) order, §4.2
// alignment and padding, §4.3 bucket_size and the cut rule, §5 param_index_map and the
// bucket-relative param_to_index.  Pure host code: no CUDA call, no allocation on the
// device.
#include <cstdint>
#include <algorithm>
#include <numeric>
#include <vector>

#include "gtp.h"
#include "status.h"

namespace {

struct Key {
  int32_t param_dtype, grad_dtype, is_expert_parallel, is_layer_wise;
  bool operator==(const Key &o) const {
    return param_dtype == o.param_dtype && grad_dtype == o.grad_dtype &&
           is_expert_parallel == o.is_expert_parallel && is_layer_wise == o.is_layer_wise;
  }
};

int64_t round_up(int64_t x, int64_t d) { return (x + d - 1) / d * d; }

struct PlacedBucket {
  int32_t buffer_id;
  int64_t offset, numel_unpadded, numel;
  std::vector<int32_t> params;
};

}  // namespace

extern "C" gtp_status gtp_buffer_layout(const gtp_param_desc *params, int32_t n_params,
                                        const gtp_layout_config *cfg, gtp_param_index *index,
                                        gtp_buffer_desc *buffers, int32_t *n_buffers,
                                        gtp_bucket_desc *buckets, int32_t *n_buckets) {
  gtp::clear_error();
  if (!cfg || !n_buffers || !n_buckets) return gtp::fail(GTP_E_ARG, "null cfg or count pointer");
  if (n_params < 0) return gtp::fail(GTP_E_ARG, "n_params < 0");
  if (n_params > 0 && !params) return gtp::fail(GTP_E_ARG, "null params");
  if (cfg->dp_size < 1) return gtp::fail(GTP_E_ARG, "dp_size must be >= 1");
  const int32_t cap_buffers = *n_buffers, cap_buckets = *n_buckets;
  if (cap_buffers < 0 || cap_buckets < 0) return gtp::fail(GTP_E_ARG, "negative capacity");
  if ((cap_buffers > 0 && !buffers) || (cap_buckets > 0 && !buckets))
    return gtp::fail(GTP_E_ARG, "capacity given with a null array");

  const int64_t kMaxNumel = int64_t(1) << 50;
  for (int32_t i = 0; i < n_params; ++i) {
    const gtp_param_desc &p = params[i];
    if (p.numel <= 0 || p.numel > kMaxNumel)
      return gtp::fail(GTP_E_ARG, "param %d: numel %lld out of (0, 2^50]", i, (long long)p.numel);
    if (p.dtype != GTP_F32 && p.dtype != GTP_BF16 && p.dtype != GTP_F16)
      return gtp::fail(GTP_E_DTYPE, "param %d: dtype %d is not F32/BF16/F16", i, p.dtype);
    if (p.reserved != 0) return gtp::fail(GTP_E_ARG, "param %d: reserved field must be 0", i);
  }

  const bool distopt = cfg->use_distributed_optimizer != 0;
  const bool bucketed = cfg->bucket_size > 0;
  int64_t divisor = 1;  // bucket-end padding divisor (§4.2)
  if (distopt) {
    divisor = std::lcm<int64_t>(cfg->dp_size, 128);
    if (cfg->pad_buckets_for_high_nccl_busbw) divisor = std::lcm<int64_t>(divisor, 65536);
  }

  // §3: one buffer per distinct BufferKey, keys in order of first appearance.
  std::vector<Key> keys;
  std::vector<std::vector<int32_t>> members;
  for (int32_t i = 0; i < n_params; ++i) {
    const gtp_param_desc &p = params[i];
    Key k{p.quantized_storage ? int32_t(GTP_U8) : p.dtype,
          cfg->grad_reduce_in_fp32 ? int32_t(GTP_F32) : p.dtype, p.is_expert_parallel ? 1 : 0,
          p.is_layer_wise ? 1 : 0};
    size_t j = 0;
    while (j < keys.size() && !(keys[j] == k)) ++j;
    if (j == keys.size()) {
      keys.push_back(k);
      members.emplace_back();
    }
    members[j].push_back(i);
  }

  std::vector<int64_t> start(n_params), end(n_params);
  std::vector<int32_t> bucket_of(n_params, -1), buffer_of(n_params, -1);
  std::vector<PlacedBucket> placed;
  std::vector<int64_t> buffer_numel(keys.size());
  std::vector<int32_t> buffer_first(keys.size()), buffer_count(keys.size());

  for (size_t b = 0; b < keys.size(); ++b) {
    const int32_t buffer_id = int32_t(b);
    buffer_first[b] = int32_t(placed.size());
    int64_t bucket_start = 0, cur = 0;
    std::vector<int32_t> open;
    auto close = [&](int64_t end_unpadded) -> int64_t {
      const int64_t padded = distopt ? round_up(end_unpadded, divisor) : end_unpadded;
      PlacedBucket pb{buffer_id, bucket_start, end_unpadded - bucket_start, padded - bucket_start,
                      open};
      const int32_t bid = int32_t(placed.size());
      for (int32_t pi : open) bucket_of[pi] = bid;
      placed.push_back(std::move(pb));
      bucket_start = padded;
      open.clear();
      return padded;
    };
    const std::vector<int32_t> &mem = members[b];
    for (size_t r = mem.size(); r-- > 0;) {  // §4.1: reverse model order
      const int32_t pi = mem[r];
      const bool isolate = distopt && params[pi].is_shared_embedding;
      if (isolate && !open.empty()) cur = close(cur);
      const int64_t s = distopt ? round_up(cur, 64) : cur;  // §4.2: 64-element start
      const int64_t e = s + params[pi].numel;
      start[pi] = s;
      end[pi] = e;
      buffer_of[pi] = buffer_id;
      open.push_back(pi);
      cur = e;
      if (isolate || (bucketed && e - bucket_start >= cfg->bucket_size)) cur = close(e);  // §4.3
    }
    if (!open.empty()) cur = close(cur);
    buffer_numel[b] = cur;
    buffer_count[b] = int32_t(placed.size()) - buffer_first[b];
  }

  if (index) {
    for (int32_t i = 0; i < n_params; ++i) {
      const PlacedBucket &pb = placed[bucket_of[i]];
      index[i].start = start[i];
      index[i].end = end[i];
      index[i].start_in_bucket = start[i] - pb.offset;
      index[i].end_in_bucket = end[i] - pb.offset;
      index[i].bucket_id = bucket_of[i];
      index[i].buffer_id = buffer_of[i];
    }
  }
  const int32_t nbuf = int32_t(keys.size()), nbkt = int32_t(placed.size());
  *n_buffers = nbuf;
  *n_buckets = nbkt;
  if (buffers && cap_buffers >= nbuf) {
    for (int32_t b = 0; b < nbuf; ++b) {
      buffers[b].numel = buffer_numel[b];
      buffers[b].param_dtype = keys[b].param_dtype;
      buffers[b].grad_dtype = keys[b].grad_dtype;
      buffers[b].is_expert_parallel = keys[b].is_expert_parallel;
      buffers[b].is_layer_wise = keys[b].is_layer_wise;
      buffers[b].first_bucket = buffer_first[b];
      buffers[b].num_buckets = buffer_count[b];
    }
  }
  if (buckets && cap_buckets >= nbkt) {
    for (int32_t k = 0; k < nbkt; ++k) {
      buckets[k].offset = placed[k].offset;
      buckets[k].numel_unpadded = placed[k].numel_unpadded;
      buckets[k].numel = placed[k].numel;
      buckets[k].buffer_id = placed[k].buffer_id;
      buckets[k].num_params = int32_t(placed[k].params.size());
    }
  }
  if ((buffers || cap_buffers) && cap_buffers < nbuf)
    return gtp::fail(GTP_E_CAPACITY, "buffers capacity %d < %d", cap_buffers, nbuf);
  if ((buckets || cap_buckets) && cap_buckets < nbkt)
    return gtp::fail(GTP_E_CAPACITY, "buckets capacity %d < %d", cap_buckets, nbkt);
  return GTP_OK;
}

// The distributed optimizer's view of one dp rank: "05 · grad/param buffer ..." §6.5 (each
// rank owns the dp_rank-th equal shard of every bucket, cut without regard to parameter
// boundaries) and "Megatron-LM architecture and source guide" §6.4 (the range map built
// per parameter: the overlap of the parameter with the rank's shard).
extern "C" gtp_status gtp_shard_param_ranges(const gtp_param_index *index, int32_t n_params,
                                             const gtp_bucket_desc *buckets, int32_t n_buckets, int32_t buffer_id,
                                             int32_t dp_size, int32_t dp_rank, gtp_shard_range *out,
                                             int32_t *n_out) {
  gtp::clear_error();
  if (!n_out) return gtp::fail(GTP_E_ARG, "null n_out");
  if (n_params < 0 || n_buckets < 0) return gtp::fail(GTP_E_ARG, "negative count");
  if ((n_params > 0 && !index) || (n_buckets > 0 && !buckets)) return gtp::fail(GTP_E_ARG, "null array");
  if (dp_size < 1 || dp_rank < 0 || dp_rank >= dp_size) return gtp::fail(GTP_E_ARG, "dp_rank outside [0, dp_size)");
  const int32_t cap = *n_out;
  if (cap < 0 || (cap > 0 && !out)) return gtp::fail(GTP_E_ARG, "bad capacity");
  // parameters of each bucket of this buffer, in position order
  std::vector<std::vector<int32_t>> members(static_cast<size_t>(n_buckets));
  for (int32_t i = 0; i < n_params; ++i) {
    const gtp_param_index &x = index[i];
    if (x.buffer_id != buffer_id) continue;
    if (x.bucket_id < 0 || x.bucket_id >= n_buckets) return gtp::fail(GTP_E_RANGE, "param %d: bucket id", i);
    members[size_t(x.bucket_id)].push_back(i);
  }
  int32_t count = 0;
  for (int32_t k = 0; k < n_buckets; ++k) {
    const gtp_bucket_desc &b = buckets[k];
    if (b.buffer_id != buffer_id) continue;
    if (b.numel % dp_size) return gtp::fail(GTP_E_SHAPE, "bucket %d: numel %lld not divisible by dp %d", k,
                                            (long long)b.numel, dp_size);
    const int64_t shard = b.numel / dp_size;
    const int64_t s0 = b.offset + int64_t(dp_rank) * shard, s1 = s0 + shard;
    std::vector<int32_t> &m = members[size_t(k)];
    std::sort(m.begin(), m.end(), [&](int32_t a, int32_t c) { return index[a].start < index[c].start; });
    for (int32_t i : m) {
      const int64_t lo = std::max(index[i].start, s0), hi = std::min(index[i].end, s1);
      if (lo >= hi) continue;
      if (out && count < cap)
        out[count] = gtp_shard_range{i, k, lo, hi, lo - b.offset, lo - s0, lo - index[i].start};
      ++count;
    }
  }
  *n_out = count;
  if ((out || cap) && cap < count) return gtp::fail(GTP_E_CAPACITY, "ranges capacity %d < %d", cap, count);
  return GTP_OK;
}
