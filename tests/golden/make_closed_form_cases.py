"""Writes closed_form_cases.json: hand-derived closed forms of the sampler step.

Every value below is derived by hand from the definitions (softmax over the vocabulary,
entropy in nats, s = softmax(logits / T) . E, and the lock / re-noise rule readings); the
script only evaluates those closed forms with ``math``. It calls no implementation of the
sampler -- neither the oracle nor the CUDA library.

Run from the repository root:  python tests/golden/make_closed_form_cases.py
"""
import json
import math
import os

ln2 = math.log(2)
cases = []
cases.append(dict(
    name="three_tokens_T1", E=[[1.0], [0.0], [-1.0]], H=[[ln2]], T=1.0,
    derivation="y=(ln2,0,-ln2); exp(y-m)=(1,1/2,1/4); l=7/4; p=(4/7,2/7,1/7); s=4/7-1/7=3/7; "
               "entropy=-sum p ln p = ln7-(10/7)ln2; argmax=0",
    p=[4 / 7, 2 / 7, 1 / 7], s=[3 / 7], entropy=math.log(7) - 10 / 7 * ln2, argmax=0, pmax=4 / 7))
l2 = 1.5 + 2 ** -0.5
cases.append(dict(
    name="three_tokens_T2", E=[[1.0], [0.0], [-1.0]], H=[[ln2]], T=2.0,
    derivation="y=(ln2/2,0,-ln2/2); exp(y-m)=(1,2^-1/2,1/2); l=3/2+2^-1/2; s=(1-1/2)/l; "
               "entropy=ln l+(ln2/2)(2^-1/2)/l+ln2(1/2)/l",
    p=[1 / l2, 2 ** -0.5 / l2, 0.5 / l2], s=[0.5 / l2],
    entropy=math.log(l2) + (ln2 / 2) * (2 ** -0.5) / l2 + ln2 * 0.5 / l2, argmax=0, pmax=1 / l2))
a = 1.25
p1 = 1 / (1 + math.exp(-a))
cases.append(dict(
    name="two_tokens_identity", E=[[1.0, 0.0], [0.0, 1.0]], H=[[a, 0.0]], T=1.0,
    derivation="y=(a,0); p1=1/(1+e^-a); s=(p1,1-p1); entropy=-p1 ln p1-(1-p1)ln(1-p1)",
    p=[p1, 1 - p1], s=[p1, 1 - p1], entropy=-p1 * math.log(p1) - (1 - p1) * math.log(1 - p1),
    argmax=0, pmax=p1))
cases.append(dict(
    name="uniform_H_zero", E=[[1.0, 2.0], [3.0, -1.0], [-2.0, 0.5], [0.0, 0.5]], H=[[0.0, 0.0]],
    T=0.7,
    derivation="y=0 for every token; p=1/V; s=mean of E rows=(0.5,0.5); entropy=ln4; "
               "argmax=0 (lowest index on ties)",
    p=[0.25] * 4, s=[0.5, 0.5], entropy=math.log(4), argmax=0, pmax=0.25))

lock_cases = [
    dict(name="threshold", conf=[0.95, 0.2, 0.9, 0.89, 0.5, 0.99], lock=[0, 0, 0, 1, 0, 0],
         sampled=[7, 8, 9, 10, 11, 12], canvas=[1, 2, 3, 4, 5, 6], tau=0.9, step=0, max_steps=48,
         derivation="unlocked with c>=tau: 0,2,5 (3 already locked keeps its token 4); "
                    "1 and 4 re-noised",
         lock_after=[1, 0, 1, 1, 0, 1], locked_tokens={"0": 7, "2": 9, "3": 4, "5": 12},
         renoised=[1, 4], step_after=1, done_after=0),
    dict(name="forced_single_lock", conf=[0.3, 0.5, 0.5, 0.1], lock=[0, 0, 0, 0],
         sampled=[3, 4, 5, 6], canvas=[0, 0, 0, 0], tau=0.9, step=3, max_steps=48,
         derivation="no c>=tau: lock the largest c, lowest position among the tie 1,2 -> 1",
         lock_after=[0, 1, 0, 0], locked_tokens={"1": 4}, renoised=[0, 2, 3], step_after=4,
         done_after=0),
    dict(name="forced_skips_locked", conf=[0.8, 0.5, 0.7, 0.1], lock=[1, 0, 0, 0],
         sampled=[3, 4, 5, 6], canvas=[9, 0, 0, 0], tau=0.9, step=0, max_steps=48,
         derivation="position 0 is locked; among unlocked the largest c is position 2",
         lock_after=[1, 0, 1, 0], locked_tokens={"0": 9, "2": 5}, renoised=[1, 3], step_after=1,
         done_after=0),
    dict(name="last_step_commits_all", conf=[0.1, 0.2, 0.3], lock=[0, 1, 0], sampled=[5, 6, 7],
         canvas=[1, 2, 3], tau=0.9, step=47, max_steps=48,
         derivation="step+1==max_steps: every unlocked position takes its sample; done",
         lock_after=[1, 1, 1], locked_tokens={"0": 5, "1": 2, "2": 7}, renoised=[], step_after=48,
         done_after=1),
    dict(name="all_pass_done", conf=[0.99, 0.91], lock=[0, 0], sampled=[2, 3], canvas=[0, 0],
         tau=0.9, step=0, max_steps=48, derivation="both pass the threshold; all locked -> done",
         lock_after=[1, 1], locked_tokens={"0": 2, "1": 3}, renoised=[], step_after=1,
         done_after=1),
]

# The pages' default sampler (sokufu.com "A diffusion language model refines 256 tokens in 12
# steps", Table 2): accept from lowest to highest entropy until the 0.1 budget is spent (at
# least one), re-noise the rest; stop on mean entropy < 0.005 with unchanged argmax.
entropy_budget_cases = [
    dict(name="budget_prefix", entropy=[0.05, 0.01, 0.2, 0.03], argmax=[4, 5, 6, 7],
         prev_argmax=[4, 5, 6, 0], sampled=[8, 9, 10, 11], canvas=[0, 0, 0, 0], step=2,
         max_steps=48, budget=0.1, stop_entropy=0.005,
         derivation="ascending: 0.01 (1), 0.03 (3), 0.05 (0), 0.2 (2); running sums 0.01, 0.04, "
                    "0.09, 0.29 -> accept 1, 3, 0; position 2 re-noised",
         lock_after=[1, 1, 0, 1], accepted_tokens={"0": 8, "1": 9, "3": 11}, renoised=[2],
         step_after=3, done_after=0),
    dict(name="at_least_one", entropy=[0.5, 0.3, 0.9], argmax=[1, 2, 3], prev_argmax=[1, 2, 3],
         sampled=[4, 5, 6], canvas=[0, 0, 0], step=1, max_steps=48, budget=0.1,
         stop_entropy=0.005, derivation="the lowest entropy alone exceeds the budget: accept it",
         lock_after=[0, 1, 0], accepted_tokens={"1": 5}, renoised=[0, 2], step_after=2,
         done_after=0),
    dict(name="ties_in_position_order", entropy=[0.04, 0.04, 0.04, 0.04], argmax=[1, 1, 1, 1],
         prev_argmax=[2, 2, 2, 2], sampled=[5, 6, 7, 8], canvas=[0, 0, 0, 0], step=3,
         max_steps=48, budget=0.1, stop_entropy=0.005,
         derivation="sums 0.04, 0.08, 0.12: two accepted, equal entropies in position order",
         lock_after=[1, 1, 0, 0], accepted_tokens={"0": 5, "1": 6}, renoised=[2, 3],
         step_after=4, done_after=0),
    dict(name="stop_confident_and_stable", entropy=[0.001, 0.002, 0.0], argmax=[3, 4, 5],
         prev_argmax=[3, 4, 5], sampled=[7, 8, 9], canvas=[1, 1, 1], step=5, max_steps=48,
         budget=0.1, stop_entropy=0.005,
         derivation="mean 0.001 < 0.005 and the argmax is unchanged: the canvas takes the argmax",
         lock_after=[1, 1, 1], accepted_tokens={"0": 3, "1": 4, "2": 5}, renoised=[],
         step_after=6, done_after=1),
    dict(name="confident_but_unstable", entropy=[0.001, 0.002, 0.0], argmax=[3, 4, 5],
         prev_argmax=[3, 4, 6], sampled=[7, 8, 9], canvas=[1, 1, 1], step=5, max_steps=48,
         budget=0.1, stop_entropy=0.005,
         derivation="argmax changed: no stop; all three fit in the budget and take their samples",
         lock_after=[1, 1, 1], accepted_tokens={"0": 7, "1": 8, "2": 9}, renoised=[],
         step_after=6, done_after=0),
    dict(name="first_step_cannot_stop", entropy=[0.0, 0.0], argmax=[3, 4], prev_argmax=[3, 4],
         sampled=[7, 8], canvas=[1, 1], step=0, max_steps=48, budget=0.1, stop_entropy=0.005,
         derivation="there is no previous prediction at step 0: no stop",
         lock_after=[1, 1], accepted_tokens={"0": 7, "1": 8}, renoised=[], step_after=1,
         done_after=0),
    dict(name="last_step_takes_argmax", entropy=[0.9, 0.8], argmax=[3, 4], prev_argmax=[0, 0],
         sampled=[7, 8], canvas=[1, 1], step=47, max_steps=48, budget=0.1, stop_entropy=0.005,
         derivation="step + 1 == max_steps: the canvas takes the argmax and is done",
         lock_after=[1, 1], accepted_tokens={"0": 3, "1": 4}, renoised=[], step_after=48,
         done_after=1),
    dict(name="negative_rounding_counts_as_zero", entropy=[-1e-9, 0.2], argmax=[3, 4],
         prev_argmax=[0, 0], sampled=[7, 8], canvas=[1, 1], step=4, max_steps=48, budget=0.1,
         stop_entropy=0.005, derivation="-1e-9 counts as 0: accepted; 0.2 exceeds the budget",
         lock_after=[1, 0], accepted_tokens={"0": 7}, renoised=[1], step_after=5, done_after=0),
]

temperature_schedule = dict(
    derivation="T_k = 0.8 + (0.4 - 0.8) k / (48 - 1) (Table 2: linear from 0.8 down to 0.4)",
    t_start=0.8, t_end=0.4, max_steps=48,
    points={"0": 0.8, "47": 0.4, "23": 0.8 - 0.4 * 23 / 47, "12": 0.8 - 0.4 * 12 / 47})

doc = {
    "about": "Hand-derived closed-form cases of the sampler step (no value here comes from any "
             "implementation). Softmax, entropy and the self-conditioning vector follow "
             "DiffusionGemma Technical Report, section 6 'Sampling' (softmax over the full "
             "vocabulary; s = softmax(logits/T) . E). The lock cases follow the lock / re-noise "
             "rule readings (threshold c >= tau, at least one lock per step, sticky locks, last "
             "step commits all) of the sokufu.com article 'DiffusionGemma: Google's open "
             "diffusion LLM', section 'A diffusion language model refines 256 tokens in 12 "
             "steps', and 'Google DeepMind's DiffusionGemma Generates Text 4x Faster by "
             "Ditching Tokens', section 'How text diffusion actually works'.",
    "softmax_cases": cases,
    "lock_cases": lock_cases,
    "entropy_budget_cases": entropy_budget_cases,
    "temperature_schedule": temperature_schedule,
}
with open(os.path.join(os.path.dirname(os.path.abspath(__file__)), "closed_form_cases.json"),
          "w") as f:
    json.dump(doc, f, indent=1)
