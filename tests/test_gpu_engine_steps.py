"""Several engine steps driven by the library's host block manager on the
GPU, against the reference block manager and the oracle on the CPU: a prompt
is prefilled, forked into parallel samples that share its blocks, and
decoded token by token -- each step appends one token per sequence (the
block manager gives its slot and, when the sequence's last block is shared,
a copy-on-write pair), copies the pairs' blocks (pa_copy_blocks) before the
cache write (pa_reshape_and_cache), and attends (pa_decode_attention); a
sample finishes midway and a new request reuses its blocks.  Slots, pairs
and tables identical; pools bit-exact after every step; attention within the
contract tolerance."""
import math

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

import oracle  # noqa: E402
from oracle import block_manager as M  # noqa: E402
from stepping import assert_attention_close  # noqa: E402

H, HKV, D, BS, N, MB = 8, 2, 128, 16, 96, 16


def _bits(rng, shape):
    x = rng.standard_normal(shape, dtype=np.float32)
    return torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _dev16(a):
    return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).cuda()


@pytest.fixture(scope="module")
def B():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_cache_96_gb300 import binding
    return binding


def test_engine_steps_with_block_manager(B):
    rng = np.random.default_rng(77)
    bm, ref = B.BlockManager(N, BS, MB), M.BlockManager(N, BS, MB)
    fill = np.uint16(0x7FC0)  # bf16 NaN in every slot no token owns
    kc_o = np.full((N, BS, HKV, D), fill, np.uint16)
    vc_o = kc_o.copy()
    kc = torch.full((N, BS, HKV, D), int(np.int16(np.uint16(fill).view(np.int16))),
                    dtype=torch.int16, device="cuda").view(torch.bfloat16)
    vc = kc.clone()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    scale = 1.0 / math.sqrt(D)

    def append(seqs, counts):
        """Append tokens on both managers; write their K/V on both sides."""
        if len(seqs) == 1:
            slots, pairs = bm.append_tokens(seqs[0], counts[0])
            all_slots, all_pairs = ref.append_tokens(seqs[0], counts[0])
        else:  # one step's appends in one call
            slots, pairs = bm.append_batch(seqs, counts)
            all_slots, all_pairs = ref.append_batch(seqs, counts)
        assert slots.tolist() == all_slots and pairs == all_pairs
        T = len(all_slots)
        k, v = _bits(rng, (T, HKV, D)), _bits(rng, (T, HKV, D))
        sl = np.asarray(all_slots, np.int32)
        if all_pairs:  # copy-on-write copies come before the writes
            pm = np.asarray(all_pairs, np.int32)
            oracle.copy_blocks(kc_o, vc_o, pm)
            B.pa_copy_blocks(kc, vc, torch.from_numpy(pm).cuda(), error_word=err)
        oracle.reshape_and_cache(k, v, kc_o, vc_o, sl)
        B.pa_reshape_and_cache(_dev16(k), _dev16(v), kc, vc, torch.from_numpy(sl).cuda(),
                               error_word=err)
        return len(all_pairs)

    def attend_and_check(seqs, what):
        tables, lens = bm.build_batch(seqs, MB, N - 1)
        want_t, want_l = ref.build_batch(seqs, MB, N - 1)
        assert tables.tolist() == want_t and lens.tolist() == want_l
        q = _bits(rng, (len(seqs), H, D))
        out = torch.empty((len(seqs), H, D), dtype=torch.bfloat16, device="cuda")
        max_ctx = int(lens.max())
        ws = B.alloc_workspace(len(seqs), H, HKV, D, max_ctx, 32)
        B.pa_decode_attention(out, _dev16(q), kc, vc, torch.from_numpy(tables).cuda(),
                              torch.from_numpy(lens).cuda(), max_ctx, scale, 32, ws,
                              error_word=err)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        got_k = kc.view(torch.int16).cpu().numpy().view(np.uint16)
        got_v = vc.view(torch.int16).cpu().numpy().view(np.uint16)
        assert np.array_equal(got_k, kc_o) and np.array_equal(got_v, vc_o), what
        want = oracle.paged_attention(q, kc_o, vc_o, tables, lens, scale, oracle.BF16)
        assert_attention_close(out.float().cpu().numpy().astype(np.float64), want, what)

    # a 40-token prompt (the last block partly filled), forked into 4 samples
    for b in (bm, ref):
        b.add_sequence(0)
    append([0], [40])
    for child in (1, 2, 3):
        bm.fork(0, child)
        ref.fork(0, child)
    assert bm.ref(bm.table(0)[0]) == 4
    live = [0, 1, 2, 3]
    cows = 0
    for step in range(30):
        cows += append(live, [1] * len(live))
        attend_and_check(live, f"step {step}")
        if step == 12:  # sample 2 finishes; a new request takes blocks back
            bm.free_sequence(2)
            ref.free_sequence(2)
            live.remove(2)
            for b in (bm, ref):
                b.add_sequence(9)
            append([9], [21])
            live.append(9)
    # the first decode step of the forked samples copied their shared last block
    assert cows >= 3
    assert bm.num_free() == ref.num_free()
    bm.close()
