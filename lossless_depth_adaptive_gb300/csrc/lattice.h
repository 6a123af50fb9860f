// Host-side lattice scheduler / FSM of Depth Exploration Decoding.
//
// Follows "Depth Exploration for LLM Decoding", Algorithm 1 and section 3.2: per
// sequence, a heap-indexed binary lattice of exploration tokens (root 0, depth child
// 2i+1, position child 2i+2), an FSM state q (the round at state q creates the 2^q
// level-q nodes), validate_and_commit when the anchor D^{N-1}(0) = 2^{N-1}-1 exists,
// and the collapse onto the subtree of m = P(b_{k*}) = 2^{k*+1} with q' = N - k* - 1.
//
// Storage decisions (GPU side): every slot chain (a slot root and its depth children)
// owns one pool slot holding its hidden state and its branch KV for every layer the
// chain has computed.  The anchor path writes its KV straight into the committed
// cache; a collapse therefore only copies the new anchor chain's computed layers into
// the committed cache (one copy job) and re-indexes the survivors on the host -- the
// surviving slot chains keep their pool slots, nothing else moves.
#pragma once

#include <stdint.h>

#include <vector>

#include "../../include/dex.h"

namespace dex {

inline int heap_parent(int i) { return (i - 1) / 2; }
inline bool is_depth_child(int i) { return i > 0 && (i & 1); }
inline int heap_level(int i) {
  int l = 0;
  while ((2 << l) - 1 <= i) ++l;
  return l;
}
inline int node_stage(int i) {
  int s = 0;
  while (is_depth_child(i)) {
    ++s;
    i = heap_parent(i);
  }
  return s;
}
inline int slot_root_of(int i) {
  while (is_depth_child(i)) i = heap_parent(i);
  return i;
}

struct LatticeSeq {
  bool started = false;   // prefilled and not finished
  int p_c = 0;            // commit position (index of the next token to commit)
  int last_token = -1;    // committed token at position p_c - 1
  int q = 0;              // FSM state: the next round creates level q
  std::vector<int32_t> B;      // heap -> candidate token (-1 = not materialized)
  std::vector<int32_t> slot;   // heap (slot roots only) -> pool slot (-1)
  std::vector<int32_t> free_slots;
};

class Lattice {
 public:
  // max_branch > 0: sparse lattice -- a node is planned only when its parent exists and its
  // path holds at most max_branch position moves (the anchor chain always qualifies).
  Lattice(const int32_t* X, int n_X, int batch, bool decs, int max_branch = 0);
  int N() const { return N_; }
  int n_slots() const { return n_slots_; }
  int batch() const { return static_cast<int>(seqs_.size()); }
  const std::vector<int>& X() const { return X_; }
  int max_round_nodes() const { return batch() << (N_ - 1); }

  int start(int seq, int p_c, int last_token);
  void stop(int seq);
  bool active(int seq) const { return seqs_[seq].started; }
  int any_active() const;
  const LatticeSeq& seq(int s) const { return seqs_[s]; }

  // Plan the next round: level-q nodes of every active sequence, grouped by stage
  // (stage-major, then sequence, then heap index).  Returns the node count.
  int plan(std::vector<dex_plan_node>* out);
  // Insert the round's tokens (in plan order); commit / collapse where the anchor
  // reached the final depth.  committed[b], kstar[b] = -1 when sequence b did not commit.
  int update(const std::vector<dex_plan_node>& plan, const int32_t* tokens, int32_t* committed,
             int32_t* kstar, std::vector<dex_copy_job>* jobs);

 private:
  int alloc_slot(LatticeSeq& s);
  int N_, n_slots_;
  std::vector<int> X_;
  bool decs_;
  int max_branch_;
  std::vector<LatticeSeq> seqs_;
};

}  // namespace dex
