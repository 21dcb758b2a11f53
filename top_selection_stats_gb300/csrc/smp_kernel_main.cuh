// smp_kernel_main.cuh -- the per-row kernel (see smp_kernel.cuh for the
// pipeline overview and the helpers it uses).
#pragma once

namespace smp {

// Mask word assembly: lane l holds EPV consecutive bits; LPW lanes form one
// 32-bit word, written by the first lane of the group.
template <int DT>
__device__ __forceinline__ void store_mask_word(const Row<DT>& R, const KArgs& a, int e,
                                                uint32_t bits) {
  constexpr int EPV = 16 / (DT == DT_F32 ? 4 : 2);
  constexpr int LPW = 32 / EPV;
  const int lane = threadIdx.x & 31;
  uint32_t word = bits << (EPV * (lane % LPW));
#pragma unroll
  for (int o = 1; o < LPW; o <<= 1) word |= __shfl_xor_sync(0xffffffffu, word, o);
  const int gw = (R.base_id + e) / 32;
  if ((lane % LPW) == 0 && gw < a.W) a.kept_mask[(size_t)R.row * a.W + gw] = word;
}

// Membership bits of one vector: key > kB, or a copy of kB whose CTA-local
// rank (id order) is below inc.  tie_run carries the warp's running rank.
template <int DT>
__device__ __forceinline__ uint32_t member_bits(const float* x, uint32_t kB, int inc, bool ranked,
                                                int& tie_run) {
  constexpr int EPV = 16 / (DT == DT_F32 ? 4 : 2);
  uint32_t bits = 0u, tbits = 0u;
#pragma unroll
  for (int j = 0; j < EPV; ++j) {
    if (is_neg_inf(x[j])) continue;
    const uint32_t k = fkey(x[j]);
    if (k > kB) bits |= 1u << j;
    else if (k == kB) tbits |= 1u << j;
  }
  if (ranked) {
    const int nt = __popc(tbits);
    const int incl = warp_incl_scan(nt);
    int rr = tie_run + incl - nt;
#pragma unroll
    for (int j = 0; j < EPV; ++j)
      if ((tbits >> j) & 1u) {
        if (rr < inc) bits |= 1u << j;
        ++rr;
      }
    tie_run += __shfl_sync(0xffffffffu, incl, 31);
  } else if (inc > 0) {
    bits |= tbits;  // every copy in this CTA is kept
  }
  return bits;
}

template <int DT>
__device__ __forceinline__ void store_probs(const Row<DT>& R, const KArgs& a, int e, const float* x,
                                            uint32_t bits, bool greedy, float inv_mp) {
  constexpr int EPV = 16 / (DT == DT_F32 ? 4 : 2);
#pragma unroll
  for (int j = 0; j < EPV; ++j) {
    const int le = e + j;
    if (le < R.n_local) {
      float pr = 0.f;
      if ((bits >> j) & 1u) pr = greedy ? 1.f : weight(R, x[j]) * inv_mp;
      a.probs[(size_t)R.row * a.V + R.base_id + le] = pr;
    }
  }
}

// Output for rows whose kept set the leader already resolved (and for greedy
// rows): packed mask words and probabilities of this CTA's slice.
template <int DT>
__device__ void output_resolved(const Row<DT>& R, const KArgs& a, uint32_t kB, int inc, int cpy,
                                bool greedy, int argmax_id, double Mp) {
  constexpr int EPV = 16 / (DT == DT_F32 ? 4 : 2);
  if (!a.kept_mask && !a.probs) return;
  const bool ranked = !greedy && inc > 0 && inc < cpy;
  if (ranked) count_ties(R, kB);
  int tie_run = 0;
  for (int w = 0; w < (int)(threadIdx.x >> 5) && ranked; ++w) tie_run += R.ms->wties[w];
  const float vB = key_to_float(kB);
  const float inv_mp = greedy ? 1.f : (float)(1.0 / Mp);
  for (int it = 0; it < R.iters; ++it) {
    const int e = vec_elem(R, it);
    const uint4 r = ld_vec(R, e);
    uint32_t bits = 0u;
    float x[EPV];
    bool any;
    if (greedy) {
      const int d = argmax_id - (R.base_id + e);
      if (d >= 0 && d < EPV) bits = 1u << d;
      any = a.probs != nullptr;
      if (any) unpack<DT>(r, x);
    } else {
      any = __any_sync(0xffffffffu, vmax<DT>(r) >= vB);
      if (any) {
        unpack<DT>(r, x);
        bits = member_bits<DT>(x, kB, inc, ranked, tie_run);
      }
    }
    if (a.kept_mask) store_mask_word(R, a, e, bits);
    if (a.probs) {
      if (!any) {
#pragma unroll
        for (int j = 0; j < EPV; ++j) x[j] = 0.f;
      }
      store_probs(R, a, e, x, bits, greedy, inv_mp);
    }
  }
}

// Output for rows whose kept set was not gathered (all legal kept, or the
// full-row refinement): masks, the cluster-wide normaliser, the draw by the
// CTA holding u * M_p, and probabilities.  Writes count / token / Mp.
template <int DT>
__device__ void output_distributed(const Row<DT>& R, const KArgs& a, uint32_t kB, int inc,
                                   bool all, double u, bool sample, int& count_out) {
  constexpr int EPV = 16 / (DT == DT_F32 ? 4 : 2);
  cg::cluster_group cluster = cg::this_cluster();
  Misc* ms = R.ms;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const bool ranked = !all && inc > 0;
  if (ranked) count_ties(R, kB);
  int warp_tie0 = 0;
  for (int w = 0; w < warp && ranked; ++w) warp_tie0 += ms->wties[w];
  const float vB = all ? -INFINITY : key_to_float(kB);
  // (1) masks, per-warp member mass / count / last id
  {
    int tie_run = warp_tie0;
    float msum = 0.f;
    double wmass = 0.0;
    int cnt = 0, last = -1;
    for (int it = 0; it < R.iters; ++it) {
      const int e = vec_elem(R, it);
      const uint4 r = ld_vec(R, e);
      uint32_t bits = 0u;
      if (all || __any_sync(0xffffffffu, vmax<DT>(r) >= vB)) {
        float x[EPV];
        unpack<DT>(r, x);
        if (all) {
#pragma unroll
          for (int j = 0; j < EPV; ++j)
            if (!is_neg_inf(x[j])) bits |= 1u << j;
        } else {
          bits = member_bits<DT>(x, kB, inc, ranked, tie_run);
        }
#pragma unroll
        for (int j = 0; j < EPV; ++j)
          if ((bits >> j) & 1u) msum += weight(R, x[j]);
        if (bits) last = R.base_id + e + (31 - __clz(bits));
        cnt += __popc(bits);
      }
      if ((it & 15) == 15) {
        wmass += warp_sum((double)msum);
        msum = 0.f;
      }
      if (a.kept_mask) store_mask_word(R, a, e, bits);
    }
    wmass += warp_sum((double)msum);
    cnt = __reduce_add_sync(0xffffffffu, cnt);
    last = (int)__reduce_max_sync(0xffffffffu, (unsigned)(last + 1)) - 1;
    if (lane == 0) {
      ms->wmass[warp] = wmass;
      ms->wmem[warp] = cnt;
      ms->wlast[warp] = last;
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    XRec rec;
    double m = 0.0;
    int c = 0, l = -1;
    for (int w = 0; w < NWARP; ++w) {
      m += ms->wmass[w];
      c += ms->wmem[w];
      l = max(l, ms->wlast[w]);
    }
    rec.d[0] = m;
    rec.i[0] = c;
    rec.i[1] = l;
    ms->tmp = rec;
  }
  __syncthreads();
  push_all(R, X_OUT, ms->tmp);
  cluster.sync();
  double Mp = 0.0;
  int count = 0;
  for (int r = 0; r < R.S; ++r) {
    Mp += rec_of(R, X_OUT, r).d[0];
    count += rec_of(R, X_OUT, r).i[0];
  }
  count_out = count;
  const double T = u * Mp;
  // (2) the draw: the CTA whose prefix mass holds T, then its warp, then the lane
  if (sample) {
    int tc = -1, lastnz = -1;
    double pre = 0.0, P = 0.0, pre_last = 0.0;
    for (int r = 0; r < R.S; ++r) {
      const double mr = rec_of(R, X_OUT, r).d[0];
      if (rec_of(R, X_OUT, r).i[0] > 0) {
        lastnz = r;
        pre_last = pre;
      }
      if (tc < 0 && mr > 0.0 && pre + mr > T) {
        tc = r;
        P = pre;
      }
      pre += mr;
    }
    if (tc < 0) {
      tc = lastnz;
      P = pre_last;
    }
    if (tc == R.rank) {
      int tw = -1, lw = -1;
      double wpre = P, tbase = 0.0, lbase = P;
      for (int w = 0; w < NWARP; ++w) {
        const double mw = ms->wmass[w];
        if (ms->wmem[w] > 0) {
          lw = w;
          lbase = wpre;
        }
        if (tw < 0 && mw > 0.0 && wpre + mw > T) {
          tw = w;
          tbase = wpre;
        }
        wpre += mw;
      }
      if (tw < 0) {
        tw = lw;
        tbase = lbase;
      }
      if (warp == tw) {
        int tie_run = warp_tie0;
        double base = tbase;
        int found = -1, lastm = -1;
        for (int it = 0; it < R.iters && found < 0; ++it) {
          const int e = vec_elem(R, it);
          const uint4 r = ld_vec(R, e);
          if (!all && !__any_sync(0xffffffffu, vmax<DT>(r) >= vB)) continue;
          float x[EPV];
          unpack<DT>(r, x);
          uint32_t bits = 0u;
          if (all) {
#pragma unroll
            for (int j = 0; j < EPV; ++j)
              if (!is_neg_inf(x[j])) bits |= 1u << j;
          } else {
            bits = member_bits<DT>(x, kB, inc, ranked, tie_run);
          }
          float wl[EPV];
          float ls = 0.f;
#pragma unroll
          for (int j = 0; j < EPV; ++j) {
            wl[j] = ((bits >> j) & 1u) ? weight(R, x[j]) : 0.f;
            ls += wl[j];
          }
          const float li = warp_incl_scan(ls);
          const float tot = __shfl_sync(0xffffffffu, li, 31);
          const bool cross = (base + (double)li > T) && ls > 0.f;
          const unsigned cm = __ballot_sync(0xffffffffu, cross);
          if (bits) lastm = R.base_id + e + (31 - __clz(bits));
          lastm = (int)__reduce_max_sync(0xffffffffu, (unsigned)(lastm + 1)) - 1;
          if (cm) {
            const int fl = __ffs(cm) - 1;
            if (lane == fl) {
              double c = base + (double)(li - ls);
              int tok = -1, lastl = -1;
#pragma unroll
              for (int j = 0; j < EPV; ++j)
                if ((bits >> j) & 1u) {
                  c += (double)wl[j];
                  lastl = R.base_id + e + j;
                  if (tok < 0 && c > T) tok = lastl;
                }
              found = (tok >= 0) ? tok : lastl;
            }
            found = __shfl_sync(0xffffffffu, found, fl);
          }
          base += (double)tot;
        }
        if (lane == 0) a.tokens[R.row] = (found >= 0) ? found : lastm;
      }
    }
  }
  // (3) probabilities
  if (a.probs) {
    const float inv_mp = (float)(1.0 / Mp);
    int tie_run = warp_tie0;
    for (int it = 0; it < R.iters; ++it) {
      const int e = vec_elem(R, it);
      const uint4 r = ld_vec(R, e);
      float x[EPV];
      unpack<DT>(r, x);
      uint32_t bits = 0u;
      if (all) {
#pragma unroll
        for (int j = 0; j < EPV; ++j)
          if (!is_neg_inf(x[j])) bits |= 1u << j;
      } else {
        bits = member_bits<DT>(x, kB, inc, ranked, tie_run);
      }
      store_probs(R, a, e, x, bits, false, inv_mp);
    }
  }
}

// Walk the window members (key in [lo, hi], copies of tie_key limited to the
// first tie_inc in this CTA) -- count per warp or emit into the leader's band.
template <int DT>
__device__ int window_walk(const Row<DT>& R, uint32_t lo, uint32_t hi, uint32_t tie_key,
                           int tie_inc, bool emit, int cta_off, int cap) {
  constexpr int EPV = 16 / (DT == DT_F32 ? 4 : 2);
  cg::cluster_group cluster = cg::this_cluster();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const bool limited = tie_inc >= 0 && tie_key >= lo && tie_key <= hi;
  int tie_run = 0;
  if (limited)
    for (int w = 0; w < warp; ++w) tie_run += R.ms->wties[w];
  uint32_t* dk = emit ? cluster.map_shared_rank(R.bk, 0u) : nullptr;
  int* di = emit ? cluster.map_shared_rank(R.bi, 0u) : nullptr;
  int base = 0;
  if (emit) {
    base = cta_off;
    for (int w = 0; w < warp; ++w) base += R.ms->wcnt[0][w];
  }
  const float vlo = key_to_float(lo);
  int c = 0;
  for (int it = 0; it < R.iters; ++it) {
    const int e = vec_elem(R, it);
    const uint4 r = ld_vec(R, e);
    if (!__any_sync(0xffffffffu, vmax<DT>(r) >= vlo)) continue;
    float x[EPV];
    unpack<DT>(r, x);
    uint32_t bits = 0u, tbits = 0u;
#pragma unroll
    for (int j = 0; j < EPV; ++j) {
      if (is_neg_inf(x[j])) continue;
      const uint32_t k = fkey(x[j]);
      if (k >= lo && k <= hi) bits |= 1u << j;
      if (limited && k == tie_key) tbits |= 1u << j;
    }
    if (limited) {
      const int nt = __popc(tbits);
      const int incl = warp_incl_scan(nt);
      int rr = tie_run + incl - nt;
#pragma unroll
      for (int j = 0; j < EPV; ++j)
        if ((tbits >> j) & 1u) {
          if (rr >= tie_inc) bits &= ~(1u << j);
          ++rr;
        }
      tie_run += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (emit) {
      if (__any_sync(0xffffffffu, bits != 0u)) warp_emit(R, e, x, bits, base, dk, di, cap);
    } else {
      c += __popc(bits);
    }
  }
  if (!emit) {
    c = __reduce_add_sync(0xffffffffu, c);
    if (lane == 0) R.ms->wcnt[0][warp] = c;
    __syncthreads();
    int tot = 0;
    for (int w = 0; w < NWARP; ++w) tot += R.ms->wcnt[0][w];
    __syncthreads();
    return tot;
  }
  return 0;
}

// Gather the window into the leader's band (count, exchange offsets, emit).
// Returns the band size; per-CTA counts go to cta_cnt.
template <int DT>
__device__ int gather_window(const Row<DT>& R, uint32_t lo, uint32_t hi, uint32_t tie_key,
                             int tie_inc, int cap) {
  cg::cluster_group cluster = cg::this_cluster();
  const int cnt = window_walk(R, lo, hi, tie_key, tie_inc, false, 0, cap);
  XRec rec;
  rec.i[0] = cnt;
  push_all(R, X_GCNT, rec);
  cluster.sync();
  int off = 0, tot = 0;
  for (int r = 0; r < R.S; ++r) {
    const int cr = rec_of(R, X_GCNT, r).i[0];
    if (r < R.rank) off += cr;
    tot += cr;
  }
  window_walk(R, lo, hi, tie_key, tie_inc, true, off, cap);
  cluster.sync();
  return min(tot, cap);
}

// Leader: per-CTA copies of kB in the band and how many of them are members.
template <int DT>
__device__ void band_copies(const Row<DT>& R, int n, uint32_t kB, int* cpy, int* inc) {
  // one warp; S <= MAX_CLUSTER counters in shared memory
  const int lane = threadIdx.x & 31, ch = (n + 31) / 32;
  const int j0 = lane * ch, j1 = min(n, j0 + ch);
  if (lane < MAX_CLUSTER) {
    cpy[lane] = 0;
    inc[lane] = 0;
  }
  __syncwarp();
  for (int j = j0; j < j1; ++j) {
    if (R.bk[j] != kB) continue;
    const int id = R.bi[j] & 0x7fffffff;
    const int cta = id / R.L;
    atomicAdd(&cpy[cta], 1);
    if (!(R.bi[j] & NOT_MEMBER)) atomicAdd(&inc[cta], 1);
  }
  __syncwarp();
}

template <int DT>
__global__ void __launch_bounds__(NT, 2) smp_rows_kernel(const __grid_constant__ KArgs a) {
  constexpr int EPV = 16 / (DT == DT_F32 ? 4 : 2);
  constexpr int ES = (DT == DT_F32 ? 4 : 2);
  extern __shared__ __align__(128) char smem[];
  cg::cluster_group cluster = cg::this_cluster();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  Row<DT> R;
  R.S = (int)cluster.num_blocks();
  R.rank = (int)cluster.block_rank();
  R.row = blockIdx.x / R.S;
  R.L = a.L;
  R.base_id = R.rank * a.L;
  R.n_local = max(0, min(a.L, a.V - R.base_id));
  R.Lw = a.L / NWARP;
  R.iters = R.Lw / (32 * EPV);
  const Layout lay = make_layout(a.L, DT, a.cap, R.S);
  R.data = smem + lay.off_data;
  R.mw = reinterpret_cast<uint32_t*>(smem + lay.off_mw);
  R.lk = reinterpret_cast<uint32_t*>(smem + lay.off_lk);
  R.li = reinterpret_cast<int*>(smem + lay.off_li);
  R.bk = reinterpret_cast<uint32_t*>(smem + lay.off_bk);
  R.bi = reinterpret_cast<int*>(smem + lay.off_bi);
  R.xch = reinterpret_cast<XRec*>(smem + lay.off_xch);
  R.ms = reinterpret_cast<Misc*>(smem + lay.off_misc);
  R.has_mask = a.bitmask != nullptr;
  Misc* ms = R.ms;
  const int row = R.row;
  const bool leader = R.rank == 0;

  // ---- 1. stage the slice: bulk copies in NCHUNK pieces ------------------
  const char* src = reinterpret_cast<const char*>(a.logits) +
                    ((size_t)row * (size_t)a.ld + (size_t)R.base_id) * ES;
  const int chunk_elems = a.L / NCHUNK;
  int chunk_bulk[NCHUNK];
  int tail0 = 0;
#pragma unroll
  for (int c = 0; c < NCHUNK; ++c) {
    const int c0 = c * chunk_elems;
    const int ne = max(0, min(chunk_elems, R.n_local - c0));
    const int bytes = a.use_tma ? ((ne * ES) & ~15) : 0;
    chunk_bulk[c] = bytes;
    if (ne > 0) tail0 = c0 + bytes / ES;
  }
  if (a.use_tma) {
    if (tid == 0) {
#pragma unroll
      for (int c = 0; c < NCHUNK; ++c) mbar_init(&ms->mbar[c], 1u);
      fence_mbar_init();
    }
    __syncthreads();
    if (tid == 0) {
#pragma unroll
      for (int c = 0; c < NCHUNK; ++c) {
        if (chunk_bulk[c] > 0) {
          mbar_arrive_expect_tx(&ms->mbar[c], (uint32_t)chunk_bulk[c]);
          bulk_g2s(R.data + (size_t)c * chunk_elems * ES, src + (size_t)c * chunk_elems * ES,
                   (uint32_t)chunk_bulk[c], &ms->mbar[c]);
        }
      }
    }
  } else {
    tail0 = 0;
  }
  // plain loads: everything without TMA, the sub-16-byte tail with it
  for (int e = tail0 + tid; e < R.n_local; e += NT) {
    if constexpr (ES == 4) {
      reinterpret_cast<uint32_t*>(R.data)[e] = reinterpret_cast<const uint32_t*>(src)[e];
    } else {
      reinterpret_cast<unsigned short*>(R.data)[e] = reinterpret_cast<const unsigned short*>(src)[e];
    }
  }
  // padding past the row end: -inf, never legal
  for (int e = R.n_local + tid; e < a.L; e += NT) {
    if constexpr (DT == DT_F32) reinterpret_cast<uint32_t*>(R.data)[e] = 0xff800000u;
    else if constexpr (DT == DT_BF16) reinterpret_cast<unsigned short*>(R.data)[e] = 0xff80u;
    else reinterpret_cast<unsigned short*>(R.data)[e] = 0xfc00u;
  }
  if (R.has_mask) {
    const int w0 = R.base_id / 32;
    const uint32_t* mrow = a.bitmask + (size_t)row * (size_t)a.W;
    for (int i = tid; i < a.L / 32; i += NT) R.mw[i] = (w0 + i < a.W) ? mrow[w0 + i] : 0u;
  }
  __syncthreads();

  // ---- 2. row statistics --------------------------------------------------
  Stats st = stats_pass(R, a, chunk_bulk);
  {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ox = __shfl_xor_sync(0xffffffffu, st.bx, o);
      const int oid = __shfl_xor_sync(0xffffffffu, st.bid, o);
      argmax_combine(st.bx, st.bid, ox, oid);
    }
    const int vi[5] = {st.nl, st.nonfin, st.timeout, st.ns, 0};
    const double vd[2] = {(double)st.s, (double)st.s2};
    if (lane == 0) {
      ms->rf[warp] = st.bx;
      ms->wlast[warp] = st.bid;
    }
    XRec rec;
    block_reduce_rec(R, vi, 4, vd, 2, rec);
    float bx = ms->rf[0];
    int bid = ms->wlast[0];
    for (int w = 1; w < NWARP; ++w) argmax_combine(bx, bid, ms->rf[w], ms->wlast[w]);
    rec.i[4] = __float_as_int(bx);
    rec.i[5] = bid;
    push_all(R, X_STATS, rec);
    cluster.sync();
  }
  float gmax = -INFINITY;
  int gargmax = 0x7fffffff, nl = 0, nonfin = 0, timeout = 0, nsamp = 0;
  double sum = 0.0, sum2 = 0.0;
  for (int r = 0; r < R.S; ++r) {
    const XRec& q = rec_of(R, X_STATS, r);
    argmax_combine(gmax, gargmax, __int_as_float(q.i[4]), q.i[5]);
    nl += q.i[0];
    nonfin |= q.i[1];
    timeout |= q.i[2];
    nsamp += q.i[3];
    sum += q.d[0];
    sum2 += q.d[1];
  }

  // ---- 3. parameters and row status --------------------------------------
  const float t = a.temperature ? a.temperature[row] : 0.f;
  const int kk = a.top_k ? a.top_k[row] : 1;
  const float pp = a.top_p ? a.top_p[row] : 1.f;
  int status = ST_OK;
  if (a.mode != MODE_ARGMAX) {
    const bool bad = isnan(t) || t < 0.f || kk < 1 || isnan(pp) || !(pp > 0.f) || pp > 1.f;
    if (bad) status = ST_INVALID;
  }
  if (status == ST_OK) {
    if (timeout) status = ST_TIMEOUT;
    else if (nonfin) status = ST_NONFINITE;
    else if (nl == 0) status = ST_EMPTY;
  }
  const bool greedy = (a.mode == MODE_ARGMAX) || (t == 0.f);
  int* rinfo = a.row_info ? a.row_info + (size_t)row * 4 : nullptr;

  if (a.mode == MODE_ARGMAX || status != ST_OK) {
    if (a.mode != MODE_ARGMAX) {
      if (a.kept_mask) {
        const int w0 = R.base_id / 32, w1 = min(a.W, (R.base_id + a.L) / 32);
        for (int w = w0 + tid; w < w1; w += NT) a.kept_mask[(size_t)row * a.W + w] = 0u;
      }
      if (a.probs)
        for (int e = tid; e < R.n_local; e += NT) a.probs[(size_t)row * a.V + R.base_id + e] = 0.f;
    }
    if (leader && tid == 0) {
      if (a.tokens) a.tokens[row] = (status == ST_OK) ? gargmax : -1;
      if (a.status) a.status[row] = status;
      if (a.kept_count) a.kept_count[row] = 0;
      if (rinfo) {
        rinfo[0] = status == ST_OK ? PATH_GREEDY : PATH_ERROR;
        rinfo[1] = rinfo[2] = rinfo[3] = 0;
      }
    }
    if (timeout && a.use_tma && tid == 0)
      for (int c = 0; c < NCHUNK; ++c)
        if (chunk_bulk[c] > 0) mbar_wait_bounded(&ms->mbar[c], 0u, 4000000000ll);
    return;
  }

  // ---- 4. selection --------------------------------------------------------
  R.temp = t;
  R.gmax = gmax;
  R.m_z = greedy ? 0.f : __fdiv_rn(gmax, t);
  R.c2 = greedy ? 0.f : 1.4426950408889634f / t;
  const int K = min(min(kk, a.V), nl);
  const bool need_K = K < nl, need_P = pp < 1.f;
  const bool sample = a.mode == MODE_SAMPLE;
  const double u = (sample && !greedy)
                       ? philox_uniform(a.seed ? a.seed[row] : 0ull, a.offset ? a.offset[row] : 0ull)
                       : 0.0;
  int path, band_n = 0, sel_rounds = 0, ref_rounds = 0;
  uint32_t keyB = 0u;
  int nkeepB = 0, my_inc = 0, my_cpy = 0, count = 0, token = -1;
  double Mp = 1.0;
  bool resolved = false;

  if (greedy) {
    path = PATH_GREEDY;
    count = 1;
    token = gargmax;
    resolved = true;
  } else if (!need_K && !need_P) {
    path = PATH_ALL;
  } else {
    path = PATH_SIGMA;
    // -- sigma truncation thresholds (Qrita key design 1) --
    const double mu = nsamp ? sum / nsamp : 0.0;
    const double var = nsamp ? fmax(sum2 / nsamp - mu * mu, 0.0) : 0.0;
    const float sigma = (float)sqrt(var);
    const int Kt = need_K ? K : min(nl, a.cap / 2);
    const float q = fmaxf((float)Kt / (float)nl, 1e-30f);
    float pos = (log2f(q) + 24.f) * 4.f;
    pos = fminf(fmaxf(pos, 0.f), (float)(DTAB - 1));
    const int i0 = min((int)pos, DTAB - 2);
    const float fr = pos - (float)i0;
    const float delta = a.delta[i0] + fr * (a.delta[i0 + 1] - a.delta[i0]);
    const float t0 = (float)mu + delta * sigma;
    const float mg = 0.2f * fabsf(t0);
    float thr[NTHR] = {t0 - mg, t0 - 0.5f * mg, t0, t0 + 0.5f * mg};
    // -- one pass: counts at four thresholds, candidates >= thr[0] kept per
    //    warp in id order, fast masses when top-p alone binds --
    int cnt[NTHR] = {0, 0, 0, 0};
    float fm[NTHR] = {0.f, 0.f, 0.f, 0.f};
    float fmt = 0.f;
    int base = 0;
    uint32_t* wk = R.lk + warp * CLW;
    int* wi = R.li + warp * CLW;
    for (int it = 0; it < R.iters; ++it) {
      const int e = vec_elem(R, it);
      const uint4 r = ld_vec(R, e);
      if (need_K && !__any_sync(0xffffffffu, vmax<DT>(r) >= thr[0])) continue;
      float x[EPV];
      unpack<DT>(r, x);
      uint32_t bits = 0u;
#pragma unroll
      for (int j = 0; j < EPV; ++j) {
        if (is_neg_inf(x[j])) continue;
        float w = 0.f;
        if (!need_K) {
          w = fast_weight(R, x[j]);
          fmt += w;
        }
#pragma unroll
        for (int i = 0; i < NTHR; ++i)
          if (x[j] >= thr[i]) {
            ++cnt[i];
            if (!need_K) fm[i] += w;
          }
        if (x[j] >= thr[0]) bits |= 1u << j;
      }
      if (__any_sync(0xffffffffu, bits != 0u)) warp_emit(R, e, x, bits, base, wk, wi, CLW);
    }
    int maxw[NTHR];
#pragma unroll
    for (int i = 0; i < NTHR; ++i) {
      const int wc = __reduce_add_sync(0xffffffffu, cnt[i]);
      if (lane == 0) ms->wcnt[i][warp] = wc;
    }
    if (lane == 0) ms->wst[warp] = base;  // members seen (stored: min(base, CLW))
    const double vd[5] = {(double)fm[0], (double)fm[1], (double)fm[2], (double)fm[3], (double)fmt};
    XRec rec;
    block_reduce_rec(R, cnt, NTHR, vd, need_K ? 0 : 5, rec);
    if (need_K)
      for (int i = 0; i < 5; ++i) rec.d[i] = 0.0;
    int ovf = 0;
#pragma unroll
    for (int i = 0; i < NTHR; ++i) {
      maxw[i] = 0;
      for (int w = 0; w < NWARP; ++w) maxw[i] = max(maxw[i], ms->wcnt[i][w]);
      rec.i[4 + i] = maxw[i];
    }
    for (int w = 0; w < NWARP; ++w) {
      rec.i[8 + w] = min(ms->wst[w], CLW);
      ovf |= ms->wst[w] > CLW;
    }
    rec.d[5] = (double)ovf;
    push_all(R, X_SIGMA, rec);
    cluster.sync();
    long long tcnt[NTHR] = {0, 0, 0, 0};
    int tmaxw[NTHR] = {0, 0, 0, 0};
    double tmass[NTHR] = {0.0, 0.0, 0.0, 0.0}, fMtot = 0.0;
    bool ovf_any = false;
    for (int r = 0; r < R.S; ++r) {
      const XRec& qr = rec_of(R, X_SIGMA, r);
      for (int i = 0; i < NTHR; ++i) {
        tcnt[i] += qr.i[i];
        tmaxw[i] = max(tmaxw[i], qr.i[4 + i]);
        tmass[i] += qr.d[i];
      }
      fMtot += qr.d[4];
      ovf_any |= qr.d[5] != 0.0;
    }
    const double target_fast = (double)pp * fMtot;
    int istar = -1;
    for (int i = NTHR - 1; i >= 0 && istar < 0; --i) {
      bool ok = tcnt[i] >= (need_K ? K : 1) && tcnt[i] <= a.cap;
      if (!need_K) ok = ok && tmass[i] >= target_fast * (1.0 + 1e-5);
      if (ovf_any) ok = ok && tmaxw[i] <= CLW;
      if (ok) istar = i;
    }
    if (istar >= 0) {
      // -- the band is complete: the leader pulls it and selects --
      bool filter = istar > 0;
      int xsrc = X_SIGMA, xoff = 8;
      if (ovf_any) {
        // a warp buffer overflowed at thr[0]: compact again at thr[istar]
        int b2 = 0;
        for (int it = 0; it < R.iters; ++it) {
          const int e = vec_elem(R, it);
          const uint4 r = ld_vec(R, e);
          if (!__any_sync(0xffffffffu, vmax<DT>(r) >= thr[istar])) continue;
          float x[EPV];
          unpack<DT>(r, x);
          uint32_t bits = 0u;
#pragma unroll
          for (int j = 0; j < EPV; ++j)
            if (!is_neg_inf(x[j]) && x[j] >= thr[istar]) bits |= 1u << j;
          if (__any_sync(0xffffffffu, bits != 0u)) warp_emit(R, e, x, bits, b2, wk, wi, CLW);
        }
        if (lane == 0) ms->wst[warp] = min(b2, CLW);
        __syncthreads();
        XRec r2;
        for (int w = 0; w < NWARP; ++w) r2.i[w] = ms->wst[w];
        push_all(R, X_GCNT, r2);
        cluster.sync();
        filter = false;
        xsrc = X_GCNT;
        xoff = 0;
      }
      if (leader) {
        // pull: segment (cta j, warp w) in order; one warp per segment
        const uint32_t fk = filter ? fkey(thr[istar]) : 0u;
        const int nseg = R.S * NWARP;
        if (tid == 0) {
          int acc = 0;
          for (int sg = 0; sg < nseg; ++sg) {
            ms->seg[sg] = acc;
            if (!filter) acc += rec_of(R, xsrc, sg / NWARP).i[xoff + sg % NWARP];
          }
          ms->seg[nseg] = acc;
        }
        __syncthreads();
        if (filter) {
          for (int sg = warp; sg < nseg; sg += NWARP) {
            const int j = sg / NWARP, w = sg % NWARP;
            const int ns = rec_of(R, xsrc, j).i[xoff + w];
            const uint32_t* sk = cluster.map_shared_rank(R.lk + w * CLW, (unsigned)j);
            int c = 0;
            for (int idx = lane; idx < ns; idx += 32) c += (sk[idx] >= fk) ? 1 : 0;
            c = __reduce_add_sync(0xffffffffu, c);
            if (lane == 0) ms->ri[sg % (NWARP * 16)] = c;  // nseg <= 128
          }
          __syncthreads();
          if (tid == 0) {
            int acc = 0;
            for (int sg = 0; sg < nseg; ++sg) {
              ms->seg[sg] = acc;
              acc += ms->ri[sg];
            }
            ms->seg[nseg] = acc;
          }
          __syncthreads();
        }
        for (int sg = warp; sg < nseg; sg += NWARP) {
          const int j = sg / NWARP, w = sg % NWARP;
          const int ns = rec_of(R, xsrc, j).i[xoff + w];
          const uint32_t* sk = cluster.map_shared_rank(R.lk + w * CLW, (unsigned)j);
          const int* si = cluster.map_shared_rank(R.li + w * CLW, (unsigned)j);
          int ob = ms->seg[sg];
          for (int c0 = 0; c0 < ns; c0 += 32) {
            const int idx = c0 + lane;
            const bool v = idx < ns;
            const uint32_t k = v ? sk[idx] : 0u;
            const int id = v ? si[idx] : 0;
            const bool f = v && k >= fk;
            const unsigned bal = __ballot_sync(0xffffffffu, f);
            const int p = ob + __popc(bal & ((1u << lane) - 1u));
            if (f && p < a.cap) {
              R.bk[p] = k;
              R.bi[p] = id;
            }
            ob += __popc(bal);
          }
        }
        __syncthreads();
        const int n = min(ms->seg[nseg], a.cap);
        // weights of the band, once (the leader's own local buffer is free now)
        float* bw = reinterpret_cast<float*>(R.lk);
        for (int j = tid; j < n; j += NT) bw[j] = weight(R, key_to_float(R.bk[j]));
        __syncthreads();
        int* cpyv = ms->ri;
        int* incv = ms->ri + MAX_CLUSTER;
        if (warp == 0) {
          int r1 = 0, r2 = 0;
          uint32_t kB = 0u;
          int nB = 0;
          double Mk = fMtot;
          if (need_K) {
            int ngt = 0;
            kB = warp_pivot_count(R, n, K, 0, ngt, r1);
            nB = K - ngt;
            warp_restrict(R, n, kB, nB);
            float s = 0.f;
            const int ch = (n + 31) / 32;
            for (int j = lane * ch; j < min(n, lane * ch + ch); ++j)
              if (!(R.bi[j] & NOT_MEMBER)) s += bw[j];
            Mk = warp_sum((double)s);
          }
          if (need_P) {
            const double target = (double)pp * Mk;
            double agt = 0.0;
            int copies = 0;
            const uint32_t kp = warp_pivot_mass(R, bw, n, target, 0.0, agt, copies, r2);
            nB = topp_copies(agt, (double)weight(R, key_to_float(kp)), target, copies);
            kB = kp;
            warp_restrict(R, n, kB, nB);
          }
          // kept set: members of the band, in id order
          const int ch = (n + 31) / 32;
          const int j0 = lane * ch, j1 = min(n, j0 + ch);
          double ls = 0.0;
          int lc = 0;
          for (int j = j0; j < j1; ++j)
            if (!(R.bi[j] & NOT_MEMBER)) {
              ls += (double)bw[j];
              ++lc;
            }
          double incl = ls;
#pragma unroll
          for (int o = 1; o < 32; o <<= 1) {
            const double nv = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += nv;
          }
          const double mp = __shfl_sync(0xffffffffu, incl, 31);
          const int cnt_all = __reduce_add_sync(0xffffffffu, lc);
          int tok = -1;
          if (sample) {
            const double T = u * mp;
            const bool cross = incl > T && lc > 0;
            const unsigned cm = __ballot_sync(0xffffffffu, cross);
            int fl = cm ? __ffs(cm) - 1 : -1;
            if (fl < 0) {  // rounding: the last member
              const unsigned nz = __ballot_sync(0xffffffffu, lc > 0);
              fl = 31 - __clz(nz);
            }
            if (lane == fl) {
              double c = incl - ls;
              int lastl = -1;
              for (int j = j0; j < j1; ++j)
                if (!(R.bi[j] & NOT_MEMBER)) {
                  c += (double)bw[j];
                  lastl = R.bi[j];
                  if (tok < 0 && c > T) tok = R.bi[j];
                }
              if (tok < 0) tok = lastl;
            }
            tok = __shfl_sync(0xffffffffu, tok, fl);
          }
          band_copies(R, n, kB, cpyv, incv);
          if (lane == 0) {
            XRec rr;
            rr.i[0] = (int)kB;
            rr.i[1] = nB;
            rr.i[2] = tok;
            rr.i[3] = cnt_all;
            rr.i[4] = r1 + r2;
            rr.i[5] = n;
            rr.d[0] = mp;
            ms->tmp = rr;
          }
        }
        __syncthreads();
        // per-CTA record: the common result plus that CTA's copies of kB
        if (tid < R.S) {
          XRec rr = ms->tmp;
          rr.i[6] = cpyv[tid];
          rr.i[7] = incv[tid];
          XRec* dst = cluster.map_shared_rank(R.xch + X_RES * R.S + 0, (unsigned)tid);
          *dst = rr;
        }
      }
      cluster.sync();
      const XRec& res = rec_of(R, X_RES, 0);
      keyB = (uint32_t)res.i[0];
      nkeepB = res.i[1];
      token = res.i[2];
      count = res.i[3];
      sel_rounds = res.i[4];
      band_n = res.i[5];
      my_cpy = res.i[6];
      my_inc = res.i[7];
      Mp = res.d[0];
      resolved = true;
    } else {
      // -- exact multi-pivot refinement over the whole row --
      path = PATH_FULL;
      int xr = 0;  // alternates X_REF0 / X_REF1
      uint32_t piv[NPIV + 1];
      uint32_t keyK = 0u;
      int nkeepK = 0, incK = 0;
      const uint32_t kmax = fkey(gmax);
      // per-CTA counts of the current window (for tie offsets)
      int wcc[MAX_CLUSTER];
      if (need_K) {
        Win Wd;
        int i = NTHR - 1;
        while (i >= 0 && tcnt[i] < K) --i;
        if (i >= 0) {
          Wd.lo = fkey(thr[i]);
          Wd.hi = (i < NTHR - 1) ? fkey(thr[i + 1]) - 1u : kmax;
          Wd.above_cnt = (i < NTHR - 1) ? tcnt[i + 1] : 0;
          for (int r = 0; r < R.S; ++r) {
            const XRec& qr = rec_of(R, X_SIGMA, r);
            wcc[r] = qr.i[i] - ((i < NTHR - 1) ? qr.i[i + 1] : 0);
          }
        } else {
          Wd.lo = KEY_MIN;
          Wd.hi = fkey(thr[0]) - 1u;
          Wd.above_cnt = tcnt[0];
          for (int r = 0; r < R.S; ++r)
            wcc[r] = rec_of(R, X_STATS, r).i[0] - rec_of(R, X_SIGMA, r).i[0];
        }
        Wd.hi = min(Wd.hi, kmax);
        if (Wd.hi < Wd.lo) Wd.hi = Wd.lo;
        Wd.above_mass = 0.0;
        Wd.n_in = 0;
        for (int r = 0; r < R.S; ++r) Wd.n_in += wcc[r];
        double no_target = 0.0;
        for (int g = 0; g < 12 && Wd.n_in > a.cap && Wd.lo < Wd.hi; ++g) {
          refine_pass(R, Wd, X_REF0 + xr, false, (long long)K, no_target, 0.0, 0u, -1, 0.f, piv);
          for (int r = 0; r < R.S; ++r) {
            const XRec& qr = rec_of(R, X_REF0 + xr, r);
            wcc[r] = qr.i[Wd.sub] - ((Wd.sub < NPIV) ? qr.i[Wd.sub + 1] : 0);
          }
          xr ^= 1;
          ++ref_rounds;
        }
        if (Wd.n_in <= a.cap && Wd.n_in > 0 && Wd.lo < Wd.hi) {
          const int n = gather_window(R, Wd.lo, Wd.hi, 0u, -1, a.cap);
          band_n = n;
          if (leader) {
            int* cpyv = ms->ri;
            int* incv = ms->ri + MAX_CLUSTER;
            if (warp == 0) {
              int ngt = 0, r1 = 0;
              const uint32_t kK = warp_pivot_count(R, n, K, (int)Wd.above_cnt, ngt, r1);
              const int nK = K - ngt;
              warp_restrict(R, n, kK, nK);
              band_copies(R, n, kK, cpyv, incv);
              if (lane == 0) {
                XRec rr;
                rr.i[0] = (int)kK;
                rr.i[1] = nK;
                rr.i[4] = r1;
                ms->tmp = rr;
              }
            }
            __syncthreads();
            if (tid < R.S) {
              XRec rr = ms->tmp;
              rr.i[6] = cpyv[tid];
              rr.i[7] = incv[tid];
              XRec* dst = cluster.map_shared_rank(R.xch + X_RES * R.S + 0, (unsigned)tid);
              *dst = rr;
            }
          }
          cluster.sync();
          const XRec& res = rec_of(R, X_RES, 0);
          keyK = (uint32_t)res.i[0];
          nkeepK = res.i[1];
          sel_rounds += res.i[4];
          incK = res.i[7];
          my_cpy = res.i[6];
        } else {
          // one key holds the k-th position: its copies are taken in id order
          keyK = Wd.lo;
          nkeepK = K - (int)Wd.above_cnt;
          int off = 0;
          for (int r = 0; r < R.rank; ++r) off += wcc[r];
          incK = max(0, min(wcc[R.rank], nkeepK - off));
          my_cpy = wcc[R.rank];
        }
      }
      keyB = keyK;
      nkeepB = nkeepK;
      my_inc = incK;
      if (need_P) {
        Win Wd;
        int i = NTHR - 1;
        if (!need_K) {
          while (i >= 0 && !(tmass[i] >= target_fast * (1.0 + 1e-5))) --i;
        } else {
          i = -1;
        }
        Wd.lo = need_K ? keyK : ((i >= 0) ? fkey(thr[i]) : KEY_MIN);
        Wd.hi = kmax;
        if (Wd.hi < Wd.lo) Wd.lo = Wd.hi;
        Wd.above_cnt = 0;
        Wd.above_mass = 0.0;
        Wd.n_in = 0x7fffffffffffll;
        // the target is p * M_k: with top-k binding M_k is the mass of the
        // first window (all of S_k), set inside the first pass; otherwise the
        // (fast) whole-row mass
        double target = (double)pp * fMtot;
        const float w_tie = need_K ? weight(R, key_to_float(keyK)) : 0.f;
        const int tie_inc = need_K ? incK : -1;
        for (int g = 0; g < 12 && (g == 0 || (Wd.n_in > a.cap && Wd.lo < Wd.hi)); ++g) {
          refine_pass(R, Wd, X_REF0 + xr, true, 0, target, (g == 0 && need_K) ? (double)pp : 0.0,
                      keyK, tie_inc, w_tie, piv);
          for (int r = 0; r < R.S; ++r) {
            const XRec& qr = rec_of(R, X_REF0 + xr, r);
            wcc[r] = qr.i[Wd.sub] - ((Wd.sub < NPIV) ? qr.i[Wd.sub + 1] : 0);
          }
          xr ^= 1;
          ++ref_rounds;
        }
        if (Wd.n_in <= a.cap && Wd.n_in > 0 && Wd.lo < Wd.hi) {
          if (need_K) count_ties(R, keyK);  // per-warp offsets for the limited copies
          const int n = gather_window(R, Wd.lo, Wd.hi, keyK, tie_inc, a.cap);
          band_n = n;
          if (leader) {
            int* cpyv = ms->ri;
            int* incv = ms->ri + MAX_CLUSTER;
            float* bw = reinterpret_cast<float*>(R.lk);
            for (int j = tid; j < n; j += NT) bw[j] = weight(R, key_to_float(R.bk[j]));
            __syncthreads();
            if (warp == 0) {
              double agt = 0.0;
              int copies = 0, r2 = 0;
              const uint32_t kp = warp_pivot_mass(R, bw, n, target, Wd.above_mass, agt, copies, r2);
              const int nP = topp_copies(agt, (double)weight(R, key_to_float(kp)), target, copies);
              warp_restrict(R, n, kp, nP);
              band_copies(R, n, kp, cpyv, incv);
              if (lane == 0) {
                XRec rr;
                rr.i[0] = (int)kp;
                rr.i[1] = nP;
                rr.i[4] = r2;
                ms->tmp = rr;
              }
            }
            __syncthreads();
            if (tid < R.S) {
              XRec rr = ms->tmp;
              rr.i[6] = cpyv[tid];
              rr.i[7] = incv[tid];
              XRec* dst = cluster.map_shared_rank(R.xch + X_RES * R.S + 0, (unsigned)tid);
              *dst = rr;
            }
          }
          cluster.sync();
          const XRec& res = rec_of(R, X_RES, 0);
          keyB = (uint32_t)res.i[0];
          nkeepB = res.i[1];
          sel_rounds += res.i[4];
          my_inc = res.i[7];
        } else {
          // one key holds the boundary: copies in id order by mass arithmetic
          const uint32_t kp = Wd.lo;
          const double wv = (double)weight(R, key_to_float(kp));
          long long avail_tot = 0;
          for (int r = 0; r < R.S; ++r) avail_tot += wcc[r];
          const int nP = topp_copies(Wd.above_mass, wv, target, (int)min(avail_tot, 0x7fffffffll));
          keyB = kp;
          nkeepB = nP;
          int off = 0;
          for (int r = 0; r < R.rank; ++r) off += wcc[r];
          my_inc = max(0, min(wcc[R.rank], nP - off));
        }
      }
    }
  }

  // ---- 5. outputs ------------------------------------------------------------
  if (resolved) {
    output_resolved(R, a, keyB, my_inc, my_cpy, greedy, gargmax, Mp);
  } else {
    output_distributed(R, a, keyB, my_inc, path == PATH_ALL, u, sample, count);
  }
  if (leader && tid == 0) {
    if (sample && resolved && a.tokens) a.tokens[row] = token;
    if (a.status) a.status[row] = ST_OK;
    if (a.kept_count) a.kept_count[row] = count;
    if (rinfo) {
      rinfo[0] = path;
      rinfo[1] = band_n;
      rinfo[2] = sel_rounds;
      rinfo[3] = ref_rounds;
    }
  }
}

}  // namespace smp
