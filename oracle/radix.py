"""Radix tree over token runs with KV-slot values (test infrastructure only;
see the package docstring).

What it does, after "Inside SGLang", Step 4 (Grow a prefix tree, then run out
of room) and the "SGLang" notes (RadixAttention: node contents, match_prefix,
insertion, eviction):
  * a node holds a run of token ids, the KV-pool slots of those tokens, its
    children keyed by their first token, and a lock count;
  * match_prefix walks down while the tokens agree and returns the matched
    length and the slots along the path; if the match ends inside a node, the
    node is split there, so the tree records the exact boundary; every node
    the walk passes gets a new access time;
  * insert walks the same way and adds the unmatched rest as a new leaf; it
    returns how many leading tokens were already cached (their new slots are
    duplicates the caller frees);
  * a running request locks the last node it matched, and the lock covers the
    whole path to the root; a split gives the new prefix node the lock count
    of the node it was cut from;
  * evict frees unlocked leaves in least-recently-used order; a parent that
    becomes a leaf is next in line; the root is never evicted.

Readings where the pages leave a step open: access times come from a logical
clock that advances by one for every node touched, in walk order (the walk
from the root touches ancestors first); a split prefix node takes the access
time of the node it was cut from; eviction takes the leaf with the smallest
(access time, creation number), where nodes are numbered in creation order
(root 0); an evicted leaf's slots are reported in token order.
"""
from __future__ import annotations

import heapq


class Node:
    __slots__ = ("key", "value", "children", "parent", "lock_ref", "last_access", "seq")

    def __init__(self, key, value, parent, seq, last_access):
        self.key = list(key)
        self.value = list(value)
        self.children = {}
        self.parent = parent
        self.lock_ref = 0
        self.last_access = last_access
        self.seq = seq


class RadixTree:
    def __init__(self):
        self.clock = 0
        self.next_seq = 0
        self.root = self._new_node([], [], None, 0)
        self.root.lock_ref = 1                     # the root is never evicted
        self.evictable = 0                         # tokens in unlocked nodes
        self.protected = 0                         # tokens in locked nodes

    # -------------------------------------------------------------- helpers
    def _new_node(self, key, value, parent, last_access):
        n = Node(key, value, parent, self.next_seq, last_access)
        self.next_seq += 1
        return n

    def _touch(self, node):
        self.clock += 1
        node.last_access = self.clock

    def _split(self, child, k):
        """Cut `child` after its first k tokens; returns the new prefix node."""
        parent = child.parent
        new = self._new_node(child.key[:k], child.value[:k], parent, child.last_access)
        new.lock_ref = child.lock_ref
        parent.children[child.key[0]] = new
        child.key, child.value = child.key[k:], child.value[k:]
        child.parent = new
        new.children[child.key[0]] = child
        return new

    def _walk(self, tokens):
        """Follow `tokens` as far as they match; split where a match ends inside
        a node.  Returns (last node, matched length, slots)."""
        node, pos, slots = self.root, 0, []
        self._touch(node)
        while pos < len(tokens) and tokens[pos] in node.children:
            child = node.children[tokens[pos]]
            k = 0
            while k < len(child.key) and pos + k < len(tokens) and child.key[k] == tokens[pos + k]:
                k += 1
            if k < len(child.key):
                child = self._split(child, k)
            self._touch(child)
            slots += child.value
            pos += k
            node = child
        return node, pos, slots

    # -------------------------------------------------------------- API
    def match_prefix(self, tokens):
        node, n, slots = self._walk(list(tokens))
        return n, slots, node

    def insert(self, tokens, slots):
        tokens, slots = list(tokens), list(slots)
        node, n, _ = self._walk(tokens)
        if n < len(tokens):
            leaf = self._new_node(tokens[n:], slots[n:], node, 0)
            self._touch(leaf)
            node.children[tokens[n]] = leaf
            self.evictable += len(leaf.key)
        return n

    def inc_lock_ref(self, node):
        while node is not self.root:
            if node.lock_ref == 0:
                self.evictable -= len(node.key)
                self.protected += len(node.key)
            node.lock_ref += 1
            node = node.parent

    def dec_lock_ref(self, node):
        while node is not self.root:
            if node.lock_ref == 1:
                self.evictable += len(node.key)
                self.protected -= len(node.key)
            node.lock_ref -= 1
            node = node.parent

    def evict(self, num_tokens):
        """Free at least `num_tokens` tokens (fewer if nothing more is
        evictable); returns the freed slots in eviction order."""
        heap = []

        def push_if_candidate(n):
            if n is not self.root and not n.children and n.lock_ref == 0:
                heapq.heappush(heap, (n.last_access, n.seq, id(n), n))

        stack = [self.root]
        while stack:
            n = stack.pop()
            stack.extend(n.children.values())
            push_if_candidate(n)
        freed = []
        while len(freed) < num_tokens and heap:
            _, _, _, leaf = heapq.heappop(heap)
            freed += leaf.value
            self.evictable -= len(leaf.key)
            parent = leaf.parent
            del parent.children[leaf.key[0]]
            push_if_candidate(parent)
        return freed

    def total_tokens(self):
        return self.evictable + self.protected

    def token_depth(self, node):
        """Position of the node's first token in any sequence through it."""
        d = 0
        node = node.parent
        while node is not None:
            d += len(node.key)
            node = node.parent
        return d

    def groups(self, last_nodes):
        """Shared-prefix groups of a batch whose requests matched `last_nodes`
        (one per request): every non-root node on two or more requests' paths
        is a group (start = its token depth, length = its run, members = the
        requests through it, depth = its rank on their paths).  Listed by
        (depth, start, first member)."""
        members = {}
        for r, node in enumerate(last_nodes):
            while node is not None and node is not self.root:
                members.setdefault(id(node), (node, []))[1].append(r)
                node = node.parent
        out = []
        for node, ms in members.values():
            if len(ms) < 2:
                continue
            depth, p = 0, node.parent
            while p is not self.root:
                depth, p = depth + 1, p.parent
            out.append((depth, self.token_depth(node), len(node.key), sorted(ms)))
        out.sort(key=lambda g: (g[0], g[1], g[3][0]))
        return out
