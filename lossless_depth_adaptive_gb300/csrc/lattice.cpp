// Lattice scheduler / FSM (see lattice.h) and its host-only C ABI.
#include "lattice.h"

#include <algorithm>
#include <new>

namespace dex {

Lattice::Lattice(const int32_t* X, int n_X, int batch, bool decs, int max_branch)
    : N_(n_X), n_slots_(1 << (n_X - 1)), X_(X, X + n_X), decs_(decs), max_branch_(max_branch), seqs_(batch) {
  for (auto& s : seqs_) {
    s.B.assign((1 << N_) - 1, -1);
    s.slot.assign((1 << N_) - 1, -1);
  }
}

int Lattice::start(int seq, int p_c, int last_token) {
  LatticeSeq& s = seqs_[seq];
  s.started = true;
  s.p_c = p_c;
  s.last_token = last_token;
  s.q = 0;
  std::fill(s.B.begin(), s.B.end(), -1);
  std::fill(s.slot.begin(), s.slot.end(), -1);
  s.free_slots.clear();
  for (int i = n_slots_ - 1; i >= 0; --i) s.free_slots.push_back(i);
  return 0;
}

void Lattice::stop(int seq) { seqs_[seq].started = false; }

int Lattice::any_active() const {
  int n = 0;
  for (const auto& s : seqs_) n += s.started ? 1 : 0;
  return n;
}

int Lattice::alloc_slot(LatticeSeq& s) {
  if (s.free_slots.empty()) return -1;
  const int v = s.free_slots.back();
  s.free_slots.pop_back();
  return v;
}

int Lattice::plan(std::vector<dex_plan_node>* out) {
  out->clear();
  for (int st = 0; st < N_; ++st) {
    for (int b = 0; b < batch(); ++b) {
      LatticeSeq& s = seqs_[b];
      if (!s.started || st > s.q) continue;
      const int lo = (1 << s.q) - 1, hi = (1 << (s.q + 1)) - 1;
      for (int i = lo; i < hi; ++i) {
        if (node_stage(i) != st) continue;
        if (i > 0 && s.B[heap_parent(i)] < 0) continue;   // parent pruned (or never planned)
        // P-children on the path root -> i, root first (each adds one branch position)
        int pc[32];
        int npc = 0;
        for (int j = i; j > 0; j = heap_parent(j))
          if ((j & 1) == 0) pc[npc++] = j;
        std::reverse(pc, pc + npc);
        if (max_branch_ > 0 && npc > max_branch_) continue;   // sparse lattice: speculates too far ahead
        dex_plan_node nd = {};
        nd.seq = b;
        nd.heap = i;
        nd.stage = st;
        nd.plen = npc;
        nd.pos = s.p_c - 1 + npc;
        nd.c_end = s.p_c;
        nd.target_pos = s.p_c + npc;
        const int r = slot_root_of(i);
        if (r == i) {                      // a new slot chain starts here
          const int v = alloc_slot(s);
          if (v < 0) return -1;
          s.slot[i] = v;
        }
        nd.slot = s.slot[r];
        nd.kv_commit = (r == 0) ? 1 : 0;
        nd.token = (st == 0) ? (i == 0 ? s.last_token : s.B[heap_parent(i)]) : -1;
        nd.unmasked = (st == N_ - 1) ? 1 : 0;
        nd.n_prior = 0;
        if (decs_ && !nd.unmasked) {
          for (int j = i; is_depth_child(j);) {
            j = heap_parent(j);
            nd.prior[nd.n_prior++] = s.B[j];
          }
        }
        nd.n_tail = npc;
        for (int t = 0; t < npc; ++t) nd.tail[t] = s.slot[pc[t]];
        out->push_back(nd);
      }
    }
  }
  return static_cast<int>(out->size());
}

int Lattice::update(const std::vector<dex_plan_node>& plan, const int32_t* tokens, int32_t* committed,
                    int32_t* kstar, std::vector<dex_copy_job>* jobs) {
  jobs->clear();
  for (int b = 0; b < batch(); ++b) {
    committed[b] = -1;
    kstar[b] = -1;
  }
  for (size_t k = 0; k < plan.size(); ++k) seqs_[plan[k].seq].B[plan[k].heap] = tokens[k];
  std::vector<char> in_round(batch(), 0);
  for (const auto& nd : plan) in_round[nd.seq] = 1;
  for (int b = 0; b < batch(); ++b) {
    if (!in_round[b]) continue;
    LatticeSeq& s = seqs_[b];
    if (s.q < N_ - 1) {                // advance(q)
      ++s.q;
      continue;
    }
    // validate_and_commit: y = u_{N-1}; shallowest k < N-1 with u_k = y, else N-1
    const int y = s.B[(1 << (N_ - 1)) - 1];
    int ks = N_ - 1;
    for (int k = 0; k < N_ - 1; ++k)
      if (s.B[(1 << k) - 1] == y) {
        ks = k;
        break;
      }
    committed[b] = y;
    kstar[b] = ks;
    // collapse: survivors = subtree of m = 2^(k*+1), i -> i - m 2^h
    std::vector<int32_t> nB(s.B.size(), -1), nslot(s.slot.size(), -1);
    std::vector<char> keep(n_slots_, 0);
    int new_q = 0;
    if (ks < N_ - 1 && s.B[1 << (ks + 1)] >= 0) {   // (a sparse lattice may lack m: then nothing survives)
      const int m = 1 << (ks + 1);
      const int lm = heap_level(m);
      for (int i = 0; i < static_cast<int>(s.B.size()); ++i) {
        int j = i, h = 0;
        while (heap_level(j) > lm) {
          j = heap_parent(j);
          ++h;
        }
        if (j != m) continue;
        const int ni = i - m * (1 << h);
        nB[ni] = s.B[i];
        if (s.slot[i] >= 0) {
          nslot[ni] = s.slot[i];
          keep[s.slot[i]] = 1;
        }
      }
      // the new anchor chain's computed stages 0..N-k*-2 move to the committed cache
      dex_copy_job job;
      job.seq = b;
      job.slot = s.slot[m];
      job.pos = s.p_c;
      job.n_layers = X_[N_ - ks - 2];
      jobs->push_back(job);
      new_q = N_ - ks - 1;
    }
    s.free_slots.clear();
    for (int v = n_slots_ - 1; v >= 0; --v)
      if (!keep[v]) s.free_slots.push_back(v);
    s.B.swap(nB);
    s.slot.swap(nslot);
    s.q = new_q;
    s.p_c += 1;
    s.last_token = y;
  }
  return 0;
}

}  // namespace dex

// ---- host-only C ABI --------------------------------------------------------------------
struct dex_lattice {
  dex::Lattice lat;
  std::vector<dex_plan_node> plan;
  dex_lattice(const int32_t* X, int n, int b, bool d, int mb) : lat(X, n, b, d, mb) {}
};

extern "C" {

int dex_lattice_new(const int32_t* X, int32_t n_X, int32_t batch, int32_t decs, int32_t max_branch,
                    dex_lattice** out) {
  if (!X || !out || n_X < 1 || n_X > 10 || batch < 1 || batch > 64 || max_branch < 0) return DEX_EINVAL;
  for (int i = 0; i < n_X; ++i)
    if (X[i] < 1 || (i > 0 && X[i] <= X[i - 1])) return DEX_EINVAL;
  dex_lattice* l = new (std::nothrow) dex_lattice(X, n_X, batch, decs != 0, max_branch);
  if (!l) return DEX_ENOMEM;
  *out = l;
  return DEX_OK;
}

int dex_lattice_start(dex_lattice* lat, int32_t seq, int32_t p_c, int32_t last_token) {
  if (!lat || seq < 0 || seq >= lat->lat.batch() || p_c < 1) return DEX_EINVAL;
  return lat->lat.start(seq, p_c, last_token);
}

int dex_lattice_plan(dex_lattice* lat, dex_plan_node* out, int32_t max_nodes, int32_t* n_nodes) {
  if (!lat || !n_nodes) return DEX_EINVAL;
  const int n = lat->lat.plan(&lat->plan);
  if (n < 0) return DEX_ECAPACITY;
  *n_nodes = n;
  if (n > max_nodes || (n > 0 && !out)) return DEX_ECAPACITY;
  for (int i = 0; i < n; ++i) out[i] = lat->plan[i];
  return DEX_OK;
}

int dex_lattice_update(dex_lattice* lat, const int32_t* tokens, int32_t* committed, int32_t* kstar,
                       dex_copy_job* jobs, int32_t max_jobs, int32_t* n_jobs) {
  if (!lat || !committed || !kstar || !n_jobs || (!tokens && !lat->plan.empty())) return DEX_EINVAL;
  std::vector<dex_copy_job> j;
  lat->lat.update(lat->plan, tokens, committed, kstar, &j);
  lat->plan.clear();
  *n_jobs = static_cast<int32_t>(j.size());
  if (static_cast<int>(j.size()) > max_jobs || (!j.empty() && !jobs)) return DEX_ECAPACITY;
  for (size_t i = 0; i < j.size(); ++i) jobs[i] = j[i];
  return DEX_OK;
}

int dex_lattice_state(const dex_lattice* lat, int32_t seq, int32_t* q, int32_t* p_c, int32_t* slots_used) {
  if (!lat || seq < 0 || seq >= lat->lat.batch()) return DEX_EINVAL;
  const auto& s = lat->lat.seq(seq);
  if (q) *q = s.q;
  if (p_c) *p_c = s.p_c;
  if (slots_used) *slots_used = lat->lat.n_slots() - static_cast<int>(s.free_slots.size());
  return DEX_OK;
}

void dex_lattice_free(dex_lattice* lat) { delete lat; }

}  // extern "C"
