"""The process-pool form of the oracle's plain definition used by the
full-size GPU parity tests gives exactly what the oracle's trie-based decode
attention gives, for single and multi-token (causal) queries and an fp8
pool's dequantised rows."""
import numpy as np

import workloads
from oracle import attention as A
from oracle import fp8 as F8
from oracle.pakv import OracleTrie
from tests.oracle_parallel import plain_definition


def trie_of(wl):
    trie = OracleTrie(wl.chunk, 100_000)
    for sid in wl.seq_ids():
        k, v = wl.kv_rows(sid)
        if wl.kv_dtype == "fp8":
            k, v = F8.dequantize(F8.quantize(k, 1.0), 1.0), F8.dequantize(F8.quantize(v, 1.0), 1.0)
        trie.insert(sid, wl.tokens(sid), k, v)
    return trie


def test_matches_trie_decode_single_token():
    wl = workloads.make("tiny")
    q = wl.queries(3)
    batch = wl.seq_ids()[::-1]
    np.testing.assert_array_equal(plain_definition(wl, batch, q),
                                  A.decode_attention(trie_of(wl), batch, 0, q, wl.scale))


def test_matches_trie_decode_multi_token_causal_and_fp8():
    wl = workloads.make("tiny")
    wl.q_len, wl.kv_dtype = 3, "fp8"
    q = wl.queries(1)
    batch = wl.seq_ids()
    np.testing.assert_array_equal(plain_definition(wl, batch, q),
                                  A.decode_attention_multi(trie_of(wl), batch, 0, q, wl.scale, causal=True))


def test_matches_after_churn():
    wl = workloads.make("multi_tenant")
    wl.churn_step()
    batch = wl.seq_ids()[:3]
    q = wl.queries(1)[:3]
    want = np.stack([A.softmax_attention(q[i], *[x[0] for x in wl.kv_rows(s)], wl.scale)
                     for i, s in enumerate(batch)])
    np.testing.assert_array_equal(plain_definition(wl, batch, q), want)
