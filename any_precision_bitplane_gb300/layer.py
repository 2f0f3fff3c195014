"""Device-resident bitplane layers and their Weight Page Tables.

Uploads a layer's 8-bit codes and per-row LUTs, encodes the codes into the
overlay bitplane format with the library's own packing kernel, and builds the
page table (PagedWeight, "Core components" 1: one entry per linear block with
its committed bitwidth).  Memory layout in HBM, per layer:

  planes_gu  int32 [E, 8, H/32, 2I]   (raw uint32 plane words: plane, word, row)
  planes_dn  int32 [E, 8, I/32, H]
  lut_gu[b]  fp16  [E, 2I, 2^b]       for b in 3, 4, 5, 6, 8
  lut_dn[b]  fp16  [E, H, 2^b]

Block 2e points at planes_gu[e] and lut_gu[q][e]; block 2e+1 at planes_dn[e]
and lut_dn[q][e].
"""
import numpy as np
import torch

from . import BITWIDTHS, PW_PAGE_GPU, PageTable, pack_bitplanes


class DeviceLayer:
    def __init__(self, layer, device="cuda"):
        cfg = layer.cfg
        self.cfg = cfg
        self.E, self.H, self.I, self.k = cfg.E, cfg.H, cfg.I, cfg.k
        self.device = torch.device(device)
        E, H, I = self.E, self.H, self.I
        self.planes_gu = torch.empty((E, 8, H // 32, 2 * I), dtype=torch.int32, device=device)
        self.planes_dn = torch.empty((E, 8, I // 32, H), dtype=torch.int32, device=device)
        for e in range(E):
            codes = torch.from_numpy(np.ascontiguousarray(layer.codes_gu[e])).to(device)
            pack_bitplanes(codes, planes=self.planes_gu[e])
            codes = torch.from_numpy(np.ascontiguousarray(layer.codes_dn[e])).to(device)
            pack_bitplanes(codes, planes=self.planes_dn[e])
        self.lut_gu = {b: torch.from_numpy(layer.lut_gu[b]).to(device) for b in BITWIDTHS}
        self.lut_dn = {b: torch.from_numpy(layer.lut_dn[b]).to(device) for b in BITWIDTHS}
        self.q = np.array(layer.q, dtype=np.int32)
        self.table = PageTable(self.entries())
        torch.cuda.synchronize(self.device)

    def lut_ptr(self, block, q):
        e, m = divmod(int(block), 2)
        t = self.lut_gu[q] if m == 0 else self.lut_dn[q]
        return t[e].data_ptr()

    def planes_ptr(self, block):
        e, m = divmod(int(block), 2)
        return (self.planes_gu if m == 0 else self.planes_dn)[e].data_ptr()

    def entries(self):
        out = []
        for e in range(self.E):
            for m in range(2):
                b = 2 * e + m
                q = int(self.q[e, m])
                out.append((q, PW_PAGE_GPU, self.planes_ptr(b), self.lut_ptr(b, q)))
        return out

    def commit(self, block_ids, new_q, stream=None):
        """Recommit bitwidths (stream-ordered) and track them on the host."""
        luts = [self.lut_ptr(b, q) for b, q in zip(block_ids, new_q)]
        self.table.commit(block_ids, new_q, luts, stream=stream)
        for b, q in zip(block_ids, new_q):
            self.q[b // 2, b % 2] = int(q)

    def clone(self):
        """An independent copy (new planes, LUTs and page table) with the same contents."""
        c = DeviceLayer.__new__(DeviceLayer)
        c.cfg, c.E, c.H, c.I, c.k, c.device = self.cfg, self.E, self.H, self.I, self.k, self.device
        c.planes_gu = self.planes_gu.clone()
        c.planes_dn = self.planes_dn.clone()
        c.lut_gu = {b: t.clone() for b, t in self.lut_gu.items()}
        c.lut_dn = {b: t.clone() for b, t in self.lut_dn.items()}
        c.q = self.q.copy()
        c.table = PageTable(c.entries())
        return c

    def routed_bytes(self, topk_ids_np, blocks=(0, 1)):
        """Algorithmic weight bytes one forward call reads: top-q planes + committed LUT
        of every block of every routed expert (blocks: 0 = gate_up, 1 = down)."""
        total = 0
        for e in np.unique(np.asarray(topk_ids_np)):
            for m, (N, K) in enumerate(((2 * self.I, self.H), (self.H, self.I))):
                if m not in blocks:
                    continue
                q = int(self.q[e, m])
                total += q * N * K // 8 + N * (1 << q) * 2
        return total

    def close(self):
        self.table.close()
