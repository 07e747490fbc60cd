"""GPU parity of the top-k path's less common branches, against the oracle,
through the C ABI.  The rows are built so that a given branch of the
decision must run ("KV Cache 优化（四）" §4: every logit >= the k-th largest
is kept, ties included):

* a pass thread with more than four candidate groups (its four largest
  groups cannot list them all: the exact path);
* a thread with exactly three candidate groups (the third reload round);
* more than 512 listed logits in a row (ties at the threshold: the exact
  path);
* more than 1,024 candidate groups in a position (the exact path).

A group is (16 KiB chunk c of the row's body, pass thread t): the 16-byte
vectors t, t + 256, t + 512, t + 768 of the chunk, so the first element of
vector t of chunk c is token c * (16384 / element size) + t * (16 / element
size) in a row whose body starts at token 0.  Results must equal the
oracle's exactly away from boundary cases, like every sampled test.
"""
import numpy as np
import pytest
import torch

from parity import compare_chain, run_chain
from speculative_decoding_verification_37_gb300 import workloads as W

pytestmark = pytest.mark.gpu

V = 60000  # 16-byte-aligned rows for both element types; at least six chunks


def chain(dt, k, seed, B=4, gamma=2):
    s = W.ChainSpec(f"paths B={B} g={gamma} V={V} k={k}", B=B, gamma=gamma, V=V, dtype=dt,
                    target_sigma=2.0, temperature=1.0, top_k=k, draft_sigma=1.0)
    return W.make_chain(s, seed=seed)


def token(dt, c, t):
    es = 2 if dt == "bf16" else 4
    return c * (16384 // es) + t * (16 // es)


def set_values(rows, idx, values, dt):
    """rows: a 2-D tensor of logits rows; writes values at token ids idx in every row."""
    v = torch.as_tensor(np.asarray(values, np.float32)).to(rows.dtype)
    rows[:, torch.as_tensor(idx)] = v


@pytest.mark.parametrize("dt", ["bf16", "f32"])
def test_thread_with_more_than_four_candidate_groups(dt):
    batch = chain(dt, 3, seed=71)
    idx = [token(dt, c, 3) for c in range(6)]  # six groups of pass thread 3
    set_values(batch.target, idx, [20.0, 21.0, 22.0, 23.0, 24.0, 25.0], dt)
    set_values(batch.draft, idx, [19.0, 20.5, 21.5, 22.5, 23.5, 24.5], dt)
    compare_chain(batch, run_chain(batch), range(batch.spec.B))


@pytest.mark.parametrize("dt", ["bf16", "f32"])
def test_thread_with_three_candidate_groups(dt):
    batch = chain(dt, 3, seed=72)
    idx = [token(dt, c, 7) for c in range(3)]  # three groups of pass thread 7
    set_values(batch.target, idx, [20.0, 21.0, 22.0], dt)
    set_values(batch.draft, idx, [20.0, 21.5, 21.0], dt)
    compare_chain(batch, run_chain(batch), range(batch.spec.B))


@pytest.mark.parametrize("dt", ["bf16", "f32"])
def test_more_listed_logits_than_the_buffer(dt):
    batch = chain(dt, 5, seed=73)
    # 600 logits tied at the maximum, three groups each for threads 0..199
    idx = [token(dt, c, t) for t in range(200) for c in range(3)]
    set_values(batch.target, idx, [16.0] * len(idx), dt)
    compare_chain(batch, run_chain(batch), range(batch.spec.B))


@pytest.mark.parametrize("dt", ["bf16", "f32"])
def test_more_candidate_groups_than_the_list(dt):
    batch = chain(dt, 4, seed=74)
    # both rows of every position: three tied groups in every pass thread
    idx = [token(dt, c, t) for t in range(256) for c in range(3)]
    set_values(batch.target, idx, [16.0] * len(idx), dt)
    set_values(batch.draft, idx, [15.0] * len(idx), dt)
    compare_chain(batch, run_chain(batch), range(batch.spec.B))
