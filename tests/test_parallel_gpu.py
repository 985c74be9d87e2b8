"""The multi-GPU entry points on one GPU.

- head_sharded_sageattn: the blocks of heads that the ranks of a world of 2
  or 3 would take, run one after the other on this GPU, joined along the head
  axis, must equal one sageattn call over every head bit for bit (each
  (batch, head) is computed from its own values only).
- ulysses_sageattn with one rank (no process group) is sageattn itself; its
  exchanges between ranks are covered by the gloo tests on CPU.
"""

import math

import pytest
import torch

from quantized_attention_fp64_gb300 import dist, sageattn, sageattn_ex
from quantized_attention_fp64_gb300.workloads import custom, make_qkv

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("world,layout", [(2, "NHD"), (3, "NHD"), (2, "HND")])
def test_head_shards_join_to_the_single_call(sage_lib, world, layout):
    w = custom(2, 7, 2300, seed_index=610, k_offset_std=2.0)
    q, k, v = make_qkv(w, "cuda", layout)
    full = sageattn(q, k, v, tensor_layout=layout)
    parts = [dist.head_sharded_sageattn(q, k, v, r, world, tensor_layout=layout) for r in range(world)]
    torch.cuda.synchronize()
    joined = torch.cat(parts, dim=2 if layout == "NHD" else 1)
    assert torch.equal(joined, full)


def test_head_shards_causal_with_lse(sage_lib):
    w = custom(1, 5, 1500, seed_index=611, k_offset_std=2.0)
    q, k, v = make_qkv(w, "cuda")
    sm = 1.0 / math.sqrt(128.0)
    full, lse = sageattn_ex(q, k, v, is_causal=True, sm_scale=sm, return_lse=True)
    parts = [dist.head_sharded_sageattn(q, k, v, r, 2, is_causal=True, sm_scale=sm, return_lse=True)
             for r in range(2)]
    torch.cuda.synchronize()
    assert torch.equal(torch.cat([p[0] for p in parts], dim=2), full)
    assert torch.equal(torch.cat([p[1] for p in parts], dim=1), lse)


@pytest.mark.parametrize("layout", ["NHD", "HND"])
def test_ulysses_single_rank_is_sageattn(sage_lib, layout):
    w = custom(1, 4, 1000, seed_index=612, k_offset_std=2.0)
    q, k, v = make_qkv(w, "cuda", layout)
    assert torch.equal(dist.ulysses_sageattn(q, k, v, tensor_layout=layout), sageattn(q, k, v, tensor_layout=layout))
    out, lse = dist.ulysses_sageattn(q, k, v, tensor_layout=layout, is_causal=True, return_lse=True)
    ref, ref_lse = sageattn_ex(q, k, v, tensor_layout=layout, is_causal=True, return_lse=True)
    torch.cuda.synchronize()
    assert torch.equal(out, ref) and torch.equal(lse, ref_lse)
