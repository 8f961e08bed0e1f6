"""Write the hand-derived attention fixtures in this folder.

The pages this library follows print no worked numerical example of the attention step, so
these fixtures are tiny cases whose exact outputs follow from closed forms; each JSON file
carries its derivation and the passage that defines the rule it exercises. This script uses
only the Python ``math`` module: no oracle and no GPU code produce any expected value.

Run:  python tests/golden/make_golden.py
"""
import json
import math
import os

HERE = os.path.dirname(os.path.abspath(__file__))
P1 = '"Porting Gemma-4 (2B / 4B / 12B) to AWS Inferentia2"'
P4 = '"Gemma-4 12B on AWS Inferentia2 - Tensor-Parallel (TP=2), device prefill"'


def layer(kind, window, n_q, n_kv, d, k_eq_v=False):
    return dict(kind=kind, window=window, n_q=n_q, n_kv=n_kv, d=d, k_eq_v=k_eq_v)


def write(name, case):
    # the pin loader expects head_dim under that name
    for l in case["layers"]:
        l["head_dim"] = l.pop("d")
    with open(os.path.join(HERE, name), "w") as f:
        json.dump(case, f, indent=1)
        f.write("\n")


def logistic(x):
    return 1.0 / (1.0 + math.exp(-x))


def main():
    # 1. two keys: weights are the logistic of the score difference
    w0 = logistic(0.5 * 2.0 - 0.0)
    write("two_keys_logistic.json", dict(
        source=f"{P1}, section 4.3 (eager attention: matmul, softmax, matmul)",
        derivation="scale 0.5, q=(1,0,0,0), k0=(2,0,0,0), k1=0: s0=1, s1=0; "
                   "w0=1/(1+e^-1), w1=1-w0; v0=e_0, v1=e_1 so o=(w0, w1, 0, 0)",
        layers=[layer(1, 0, 1, 1, 4)], owner_map=[0], layer=0, scale=0.5, seq_lens=[2],
        q=[[[[1, 0, 0, 0]]]],
        k_cache={"0": [[[[2, 0, 0, 0], [0, 0, 0, 0]]]]},
        v_cache={"0": [[[[1, 0, 0, 0], [0, 1, 0, 0]]]]},
        expected=[[[[w0, 1.0 - w0, 0.0, 0.0]]]], tol=1e-15))

    # 2. sliding window of 2 keys in a 2-token prefill: equal weights over {p-1, p}
    write("sliding_window_prefill.json", dict(
        source=f"{P1}, model family table (sliding_window) and section 2.3 (sliding + global)",
        derivation="K=0 gives equal weights over the attended keys; W=2, len=5, two queries at "
                   "p=3 and p=4 attend {2,3} and {3,4}; v_j=(j, 10j) so o=(2.5,25) and (3.5,35)",
        layers=[layer(0, 2, 1, 1, 2)], owner_map=[0], layer=0, scale=1.0, seq_lens=[5],
        q=[[[[0.5, -1.0]], [[2.0, 3.0]]]],
        k_cache={"0": [[[[0, 0] for _ in range(5)]]]},
        v_cache={"0": [[[[j, 10 * j] for j in range(5)]]]},
        expected=[[[[2.5, 25.0]], [[3.5, 35.0]]]], tol=1e-15))

    # 3. GQA grouping: query heads 0,1 read KV head 0; heads 2,3 read KV head 1
    write("gqa_groups.json", dict(
        source=f"{P1}, section 2.2 (repeat_kv broadcasts each KV head to a group of query heads)",
        derivation="n_q=4, n_kv=2 so groups of G=2 consecutive query heads; K=0, every value of "
                   "KV head 0 is 10 and of KV head 1 is 20, so heads 0,1 give 10 and 2,3 give 20",
        layers=[layer(1, 0, 4, 2, 1)], owner_map=[0], layer=0, scale=1.0, seq_lens=[3],
        q=[[[[1.0], [2.0], [3.0], [4.0]]]],
        k_cache={"0": [[[[0.0]] * 3, [[0.0]] * 3]]},
        v_cache={"0": [[[[10.0]] * 3, [[20.0]] * 3]]},
        expected=[[[[10.0], [10.0], [20.0], [20.0]]]], tol=1e-15))

    # 4. cross-layer sharing: layer 1 reads layer 0's cache
    write("shared_owner.json", dict(
        source=f"{P1}, section 2.1 (shared layers attend against an earlier owner layer's K/V)",
        derivation="layer 1 has no cache of its own and owner_map[1]=0; K=0, values 1,2,3 so "
                   "the global decode query averages them: o=2",
        layers=[layer(1, 0, 1, 1, 1), layer(1, 0, 1, 1, 1)], owner_map=[0, 0], layer=1,
        scale=1.0, seq_lens=[3], q=[[[[5.0]]]],
        k_cache={"0": [[[[0.0], [0.0], [0.0]]]]},
        v_cache={"0": [[[[1.0], [2.0], [3.0]]]]},
        expected=[[[[2.0]]]], tol=1e-15))

    # 5. K as V: the output is a convex combination of the keys themselves
    w1 = logistic(1.0)
    write("k_eq_v.json", dict(
        source=f"{P4}, text config (attention_k_eq_v=true: global layers reuse K as V)",
        derivation="scale 1, q=(1,0), k0=(0,0), k1=(1,2): s0=0, s1=1, w1=1/(1+e^-1); V=K so "
                   "o = w1*(1,2)",
        layers=[layer(1, 0, 1, 1, 2, True)], owner_map=[0], layer=0, scale=1.0, seq_lens=[2],
        q=[[[[1.0, 0.0]]]],
        k_cache={"0": [[[[0.0, 0.0], [1.0, 2.0]]]]},
        expected=[[[[w1, 2.0 * w1]]]], tol=1e-15))


if __name__ == "__main__":
    main()
