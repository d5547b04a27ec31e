"""Seeded synthetic inputs for the layer step: paged pools, block tables, queries, new tokens.

This module only draws random numbers and lays them out; it performs none of the
method's arithmetic (no gating, normalisation, rotation, scoring or selection).  The
same bytes feed the CUDA library and, in the tests, the CPU oracle.

Workloads ("cases") follow the layer step of a DeepSeek-V4-style c4a / c128a layer:
each request has ``cached`` raw tokens already in the caches and appends ``new``
tokens; the queries are either the last new token of each request (decode) or every
new token (chunked prefill).  All value draws are N(0, 1) (indexer head weights
U(0, 1)); bf16 values are torch's round-to-nearest of fp32 draws; fp8 codes are
torch's e4m3 conversion of 64 * N(0, 1) draws with a per-row scale drawn
U(0.5, 1.5) / 64; fp4 indexer keys are uniformly random bytes (two e2m1 codes each, every code
equally likely) with a per-row scale drawn U(0.5, 1.5) / 6.  Physical blocks are a seeded permutation of a pool that is about
12% larger than what the requests need, so tables are shuffled and fragmented.  With the per-channel gate
the logits are N(0, 1) per raw token and channel.
"""
from dataclasses import dataclass, field
import math

import torch

BLOCK_POSITIONS = 256
WINDOW = {"c4a": (8, 4), "c128a": (128, 128)}


@dataclass
class CaseSpec:
    """Shape of one synthetic workload."""
    name: str
    kind: str = "c4a"
    cached: list = field(default_factory=lambda: [0])   # raw tokens already cached, per request
    new: list = field(default_factory=lambda: [1])      # raw tokens appended this step, per request
    queries: str = "last"                               # "last" (decode) or "all" (chunked prefill)
    heads: int = 64
    dim: int = 512
    rope_dim: int = 64
    idx_heads: int = 8                                  # 0: no indexer (c128a reads every entry)
    idx_dim: int = 128
    topk: int = 512
    window: int = 128
    main_dtype: str = "bf16"                            # "bf16" or "fp8"
    idx_dtype: str = "fp8"                              # indexer keys: "fp8" (e4m3) or "fp4" (e2m1, packed)
    gate: str = "scalar"                                # compressor logits: "scalar" (per raw token) or "channel"
    swa_dtype: str = "bf16"
    index_compress: bool = True                         # run the indexer compressor on the new tokens
    seed: int = 0

    @property
    def batch(self):
        return len(self.cached)

    @property
    def total(self):
        return [c + n for c, n in zip(self.cached, self.new)]


def _gen(seed, device):
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _randn(shape, gen, device):
    return torch.randn(shape, generator=gen, device=device, dtype=torch.float32)


def _fp8_codes_and_scale(rows, dim, gen, device):
    x = torch.clamp(_randn((rows, dim), gen, device) * 64.0, -448.0, 448.0)
    codes = x.to(torch.float8_e4m3fn).view(torch.uint8)
    scale = (torch.rand((rows,), generator=gen, device=device) + 0.5) / 64.0
    return codes, scale


def _fp4_codes_and_scale(rows, dim, gen, device):
    packed = torch.randint(0, 256, (rows, dim // 2), generator=gen, device=device, dtype=torch.int32).to(torch.uint8)
    scale = (torch.rand((rows,), generator=gen, device=device) + 0.5) / 6.0
    return packed, scale


def _tables(blocks_needed, cpu_gen, spare=0.125):
    """Block tables [B][max_blocks] (int32, -1 = unmapped) over a shuffled shared pool."""
    total = sum(len(b) for b in blocks_needed)
    num_blocks = max(1, total + int(math.ceil(total * spare)))
    perm = torch.randperm(num_blocks, generator=cpu_gen)
    max_blocks = max(1, max((max(b) + 1) if b else 1 for b in blocks_needed))
    table = torch.full((len(blocks_needed), max_blocks), -1, dtype=torch.int32)
    k = 0
    for r, blocks in enumerate(blocks_needed):
        for lb in blocks:
            table[r, lb] = int(perm[k])
            k += 1
    return table, num_blocks


def make_case(spec: CaseSpec, device="cpu"):
    """Draw every input of a case.  Returns a dict of tensors on ``device`` plus metadata."""
    dev = torch.device(device)
    cpu = _gen(spec.seed, "cpu")                 # structure: identical on every device
    gen = _gen(spec.seed + 7919, dev.type)       # values
    B, D = spec.batch, spec.dim
    w, s = WINDOW[spec.kind]
    epb = BLOCK_POSITIONS // s
    tot = spec.total

    out = {"spec": spec, "epb": epb}

    # main compressed pool: one 256-position logical block per 256 raw positions of context
    main_blocks = [list(range((t + BLOCK_POSITIONS - 1) // BLOCK_POSITIONS)) for t in tot]
    bt_main, nb_main = _tables(main_blocks, cpu)
    out["bt_main"], out["nb_main"] = bt_main.to(dev), nb_main
    if spec.main_dtype == "bf16":
        out["main_data"] = _randn((nb_main * epb, D), gen, dev).to(torch.bfloat16)
        out["main_scale"] = None
    else:
        out["main_data"], out["main_scale"] = _fp8_codes_and_scale(nb_main * epb, D, gen, dev)

    # indexer key pool (c4a only)
    if spec.idx_heads:
        bt_idx, nb_idx = _tables(main_blocks, cpu)
        out["bt_idx"], out["nb_idx"] = bt_idx.to(dev), nb_idx
        draw = _fp4_codes_and_scale if spec.idx_dtype == "fp4" else _fp8_codes_and_scale
        out["idx_data"], out["idx_scale"] = draw(nb_idx * epb, spec.idx_dim, gen, dev)

    # sliding-window pool: only blocks that some query's window or a new token touches
    if spec.queries == "last":
        first_q = [t - 1 for t in tot]
    else:
        first_q = list(spec.cached)
    swa_blocks = []
    for r in range(B):
        lo = max(0, min(first_q[r] - spec.window + 1, spec.cached[r]))
        hi = tot[r] - 1
        swa_blocks.append(list(range(lo // BLOCK_POSITIONS, hi // BLOCK_POSITIONS + 1)))
    bt_swa, nb_swa = _tables(swa_blocks, cpu)
    out["bt_swa"], out["nb_swa"] = bt_swa.to(dev), nb_swa
    if spec.swa_dtype == "bf16":
        out["swa_data"] = _randn((nb_swa * BLOCK_POSITIONS, D), gen, dev).to(torch.bfloat16)
        out["swa_scale"] = None
    else:
        out["swa_data"], out["swa_scale"] = _fp8_codes_and_scale(nb_swa * BLOCK_POSITIONS, D, gen, dev)

    # compressor rolling state: slot r holds request r's last w raw tokens (slot = pos mod w)
    out["state_slot"] = torch.arange(B, dtype=torch.int32, device=dev)
    pc = spec.gate == "channel"
    out["state_x"] = _randn((B, w, D), gen, dev).to(torch.bfloat16)
    out["state_z"] = _randn((B, w, D) if pc else (B, w), gen, dev)
    if spec.idx_heads:
        out["state_xi"] = _randn((B, w, spec.idx_dim), gen, dev).to(torch.bfloat16)
        out["state_zi"] = _randn((B, w, spec.idx_dim) if pc else (B, w), gen, dev)

    # new raw tokens (un-rotated shared-KV vectors and indexer vectors) with gate logits
    n_new = sum(spec.new)
    cu = [0]
    for n in spec.new:
        cu.append(cu[-1] + n)
    out["cu_new"] = torch.tensor(cu, dtype=torch.int32, device=dev)
    out["start_pos"] = torch.tensor(spec.cached, dtype=torch.int32, device=dev)
    out["x_new"] = _randn((n_new, D), gen, dev).to(torch.bfloat16)
    out["z_new"] = _randn((n_new, D) if pc else (n_new,), gen, dev)
    if spec.idx_heads:
        out["xi_new"] = _randn((n_new, spec.idx_dim), gen, dev).to(torch.bfloat16)
        out["zi_new"] = _randn((n_new, spec.idx_dim) if pc else (n_new,), gen, dev)

    # queries
    q_pos, q_req = [], []
    for r in range(B):
        if spec.queries == "last":
            q_pos.append(tot[r] - 1)
            q_req.append(r)
        else:
            q_pos.extend(range(spec.cached[r], tot[r]))
            q_req.extend([r] * spec.new[r])
    nq = len(q_pos)
    out["q_pos"] = torch.tensor(q_pos, dtype=torch.int32, device=dev)
    out["q_req"] = torch.tensor(q_req, dtype=torch.int32, device=dev)
    out["q"] = _randn((nq, spec.heads, D), gen, dev).to(torch.bfloat16)
    if spec.idx_heads:
        codes, scale = _fp8_codes_and_scale(nq * spec.idx_heads, spec.idx_dim, gen, dev)
        out["q8"] = codes.view(nq, spec.idx_heads, spec.idx_dim)
        out["q_scale"] = scale.view(nq, spec.idx_heads)
        out["w"] = torch.rand((nq, spec.idx_heads), generator=gen, device=dev)
    out["nq"] = nq
    out["ld"] = int(bt_main.shape[1]) * epb      # rows a score row must hold
    return out


def log_uniform_lengths(n, lo, hi, seed):
    """n context lengths floor(exp(U(ln lo, ln hi))) from a seed."""
    g = _gen(seed, "cpu")
    u = torch.rand((n,), generator=g, dtype=torch.float64)
    return [int(math.floor(math.exp(math.log(lo) + float(x) * (math.log(hi) - math.log(lo))))) for x in u]


def case_specs():
    """The five workloads at full size, keyed by name, plus the decode batch with fp4 (e2m1) indexer keys."""
    mixed = log_uniform_lengths(64, 2048, 262144, seed=1004)
    return {
        "c4a_tiny_decode": CaseSpec("c4a_tiny_decode", cached=[0], new=[4096], heads=16,
                                    idx_heads=4, idx_dim=64, index_compress=False, seed=1001),
        "c4a_decode_batch": CaseSpec("c4a_decode_batch", cached=[65535] * 32, new=[1] * 32, seed=1002),
        "c4a_decode_batch_fp4": CaseSpec("c4a_decode_batch_fp4", cached=[65535] * 32, new=[1] * 32, idx_dtype="fp4",
                                         seed=1002),
        "c128a_decode": CaseSpec("c128a_decode", kind="c128a", cached=[1048575] * 16, new=[1] * 16,
                                 idx_heads=0, topk=0, seed=1003),
        "c128a_decode_fp8": CaseSpec("c128a_decode_fp8", kind="c128a", cached=[1048575] * 16,
                                     new=[1] * 16, idx_heads=0, topk=0, main_dtype="fp8",
                                     swa_dtype="fp8", seed=1003),
        "c4a_mixed_decode": CaseSpec("c4a_mixed_decode", cached=[t - 1 for t in mixed], new=[1] * 64,
                                     seed=1004),
        "c4a_chunked_prefill": CaseSpec("c4a_chunked_prefill", cached=[131072], new=[8192],
                                        queries="all", seed=1005),
    }
