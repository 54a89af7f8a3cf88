"""GPU parity of dfv_build_tree_mask (depth and ancestor-or-self bitmask of
every draft-tree node) against the oracle's plain root walks: bit-exact over
chains, k-ary and random trees up to the 65-node limit, the lone root, and
parents outside [0, i) (treated as the root, DFV_DEV_BAD_TREE set)."""

import numpy as np
import pytest
import torch

import oracle
from tree_verify_attention_gb300 import api
from tree_verify_attention_gb300 import workload as W

from _helpers import DEV, i32_dev, need_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    need_gpu()
    from tree_verify_attention_gb300 import build
    build.build()


def _gpu_mask(parent):
    n = len(parent)
    depth = torch.full((n,), -7, dtype=torch.int32, device=DEV)
    anc = torch.full((n, api.MASK_WORDS), -7, dtype=torch.int32, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    api.build_tree_mask(i32_dev(parent), depth, anc, status=status)
    torch.cuda.synchronize()
    return depth.cpu().numpy(), anc.cpu().numpy().view(np.uint32), int(status.item())


def _oracle_mask(parent):
    n = len(parent)
    depth = oracle.tree.depths(parent)
    words = np.zeros((n, api.MASK_WORDS), dtype=np.uint32)
    for i, chain in enumerate(oracle.tree.ancestors_or_self(parent)):
        for t in chain:
            words[i, t // 32] |= np.uint32(1) << np.uint32(t % 32)
    return depth, words


def _trees():
    rng = np.random.default_rng(0)
    out = [("root", np.array([-1], dtype=np.int32))]
    for n in (2, 9, 23, 32, 33, 64, 65):
        for shape in ("chain", "kary2", "kary4", "random"):
            parent, _ = W.make_tree(rng, n, shape, max_depth=max(1, min(16, n - 1)),
                                    planted_depth=min(8, n - 1))
            out.append((f"{shape}{n}", parent))
    for k in range(8):                          # unconstrained random parents
        n = int(rng.integers(2, 66))
        parent = np.array([-1] + [int(rng.integers(0, i)) for i in range(1, n)], dtype=np.int32)
        out.append((f"uniform{k}", parent))
    return out


@pytest.mark.parametrize("name,parent", _trees(), ids=[t[0] for t in _trees()])
def test_tree_mask_matches_oracle(name, parent):
    depth, anc, status = _gpu_mask(parent)
    ref_depth, ref_anc = _oracle_mask(parent)
    assert status == 0
    assert depth.tolist() == ref_depth.tolist()
    assert np.array_equal(anc, ref_anc)


def test_tree_mask_bad_parents_become_root_children():
    parent = np.array([-1, 0, 1, 5, 2, 4, -3, 6], dtype=np.int32)   # 3 -> 5 and 6 -> -3 are bad
    depth, anc, status = _gpu_mask(parent)
    fixed = parent.copy()
    fixed[3] = 0
    fixed[6] = 0
    ref_depth, ref_anc = _oracle_mask(fixed)
    assert status & api.DEV_BAD_TREE
    assert depth.tolist() == ref_depth.tolist()
    assert np.array_equal(anc, ref_anc)


def test_tree_mask_matches_step_visibility():
    """The masks are the tree part of the attention's visibility: a chain
    tree's node i sees exactly nodes 0..i."""
    parent = np.array([-1] + list(range(64)), dtype=np.int32)
    depth, anc, _ = _gpu_mask(parent)
    assert depth.tolist() == list(range(65))
    for i in range(65):
        bits = [t for t in range(65) if (int(anc[i, t // 32]) >> (t % 32)) & 1]
        assert bits == list(range(i + 1))
